"""C-ABI boundary checks that need no GPU: the library loads, exports every
entry point the header declares, and rejects bad arguments on the host before
touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in ("moe_w4.h", "moe_w4_ablation.h")]


@pytest.fixture(scope="module")
def mw():
    from bit_quantized_sparse_gb300 import _build
    if not os.path.exists(_build.LIB):
        _build.build()
    from bit_quantized_sparse_gb300 import moe_w4
    return moe_w4


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(moe_w4_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("moe_w4_route", "moe_w4_forward_decode", "moe_w4_forward_prefill", "moe_w4_workspace_size",
              "moe_w4_strerror", "moe_w4_prepare_router", "moe_w4_router_prep_bytes", "moe_w4_set_tile_override",
              "moe_w4_ablation_prefill"):
        assert n in names


def test_library_exports_every_declared_symbol(mw):
    lib = ctypes.CDLL(mw.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), n
    assert set(declared_functions()) <= set(mw.EXPORTED)


def _layer(mw, H=2048, E=256, I=512, k=8, ptr=1 << 20):
    L = mw.MoeW4Layer()
    L.H, L.E, L.I, L.top_k = H, E, I, k
    L.router_w = L.shared_gate = ptr
    L.router_bias = None
    for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        setattr(L, n, mw.MoeW4Mat(ptr, ptr, ptr))
    return L


def test_workspace_size_host_only(mw):
    L = _layer(mw)
    w1 = mw.moe_w4_workspace_size(ctypes.byref(L), 1)
    w4k = mw.moe_w4_workspace_size(ctypes.byref(L), 4096)
    assert 0 < w1 < w4k
    # grouped activations alone: (T*k + T) rows of I and H bf16 values
    assert w4k >= (4096 * 9) * (512 + 2048) * 2
    assert mw.moe_w4_workspace_size(None, 4) == 0
    assert mw.moe_w4_status_offset() == 0


@pytest.mark.parametrize("field,val,code", [
    ("top_k", 0, -1), ("top_k", 9, -1), ("E", 0, -1), ("H", 100, -2), ("I", 192, -2), ("H", 8192, -2),
    ("E", 2048, -2), ("code_bits", 6, -2), ("code_bits", 16, -2), ("code_format", 2, -2),
    ("code_format", -1, -2), ("code_format", 1, -2)])   # E4M3 codes need code_bits = 8
def test_bad_shapes_rejected(mw, field, val, code):
    L = _layer(mw)
    setattr(L, field, val)
    assert mw.moe_w4_workspace_size(ctypes.byref(L), 8) == 0
    ws = 1 << 12
    assert mw.moe_w4_forward_prefill(ctypes.byref(L), 4, ws, ws, ws, 1 << 40, None) == code
    assert mw.moe_w4_forward_decode(ctypes.byref(L), 1, ws, ws, ws, 1 << 40, None) == code


@pytest.mark.parametrize("bits,fmt,T", [(6, 0, 1), (4, 1, 1), (0, 1, 1), (8, 2, 1), (8, 0, 2), (8, 1, 4)])
def test_noalloc_code_formats_rejected(mw, bits, fmt, T):
    """The allocation-free decode refuses code formats it has no kernels for
    (host checks only, before any device work): unknown widths or formats,
    E4M3 with 4-bit codes, and one-byte codes on a shape the one-kernel path
    does not cover (H=1024, E=128, I=256, top-4), at any T."""
    L = _layer(mw, H=1024, E=128, I=256, k=4)
    L.code_bits, L.code_format = bits, fmt
    ws = 1 << 12
    assert mw.moe_w4_forward_decode_noalloc(ctypes.byref(L), T, ws, ws, None) == mw.MOE_W4_ERR_UNSUPPORTED


def test_workspace_size_grows_with_tokens(mw):
    """The workspace a call needs never shrinks as the token count grows (a
    workspace sized for T_max serves every smaller call), for the benchmark's
    layer and a small one, across the chunk and block boundaries."""
    for shape in ((2048, 256, 512, 8), (256, 16, 128, 2)):
        L = _layer(mw, *shape)
        sizes = [mw.moe_w4_workspace_size(ctypes.byref(L), t)
                 for t in (0, 1, 2, 15, 16, 17, 127, 128, 129, 4095, 4096, 4097, 16384)]
        assert all(a <= b for a, b in zip(sizes, sizes[1:])), sizes
        assert sizes[0] > 0   # the control header and the batch-1 decode's exchange buffers


def test_token_count_cap(mw):
    """Routing and prefill take at most MOE_W4_MAX_TOKENS rows (32-bit row
    indices, at most 65535 router CTAs along the tokens): one more is refused on
    the host, before any device work, and sizes no workspace."""
    L = _layer(mw)
    p = ctypes.byref(L)
    a = 1 << 12
    big = mw.MAX_TOKENS + 1
    assert mw.moe_w4_workspace_size(p, mw.MAX_TOKENS) > 0
    assert mw.moe_w4_workspace_size(p, big) == 0
    assert mw.moe_w4_forward_prefill(p, big, a, a, a, 1 << 62, None) == mw.MOE_W4_ERR_UNSUPPORTED
    z = [a] * 7
    assert mw.moe_w4_route(p, big, a, *z, a, 1 << 62, None) == mw.MOE_W4_ERR_UNSUPPORTED
    assert mw.moe_w4_test_block_records_bytes(p, big) == 0


def test_decode_path_query(mw):
    """moe_w4_decode_path (a host query, no device work): argument checks, and
    a valid call names one of the two paths.  The row limit accepts 0..16."""
    L = _layer(mw)
    p = ctypes.c_int(-1)
    assert mw.moe_w4_decode_path(None, 2, ctypes.byref(p)) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_decode_path(ctypes.byref(L), 2, None) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_decode_path(ctypes.byref(L), 0, ctypes.byref(p)) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_decode_path(ctypes.byref(L), 17, ctypes.byref(p)) == mw.MOE_W4_ERR_UNSUPPORTED
    assert mw.moe_w4_decode_path(ctypes.byref(L), 2, ctypes.byref(p)) == mw.MOE_W4_OK
    assert p.value in (mw.MOE_W4_PATH_FUSED_ROWS, mw.MOE_W4_PATH_GROUPED)
    assert mw.moe_w4_set_decode_fused_rows(-1) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_set_decode_fused_rows(17) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_set_decode_fused_rows(0) == mw.MOE_W4_OK


def test_bad_arguments_rejected(mw):
    L = _layer(mw)
    p = ctypes.byref(L)
    a = 1 << 12
    assert mw.moe_w4_forward_prefill(None, 4, a, a, a, 1 << 40, None) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_forward_prefill(p, -1, a, a, a, 1 << 40, None) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_forward_prefill(p, 4, None, a, a, 1 << 40, None) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_forward_prefill(p, 4, a + 2, a, a, 1 << 40, None) == mw.MOE_W4_ERR_ALIGN
    assert mw.moe_w4_forward_prefill(p, 4, a, a, None, 1 << 40, None) == mw.MOE_W4_ERR_WORKSPACE
    assert mw.moe_w4_forward_prefill(p, 4, a, a, a, 1024, None) == mw.MOE_W4_ERR_WORKSPACE
    assert mw.moe_w4_forward_prefill(p, 4, a, a, a + 16, 1 << 40, None) == mw.MOE_W4_ERR_WORKSPACE
    assert mw.moe_w4_forward_decode(p, 17, a, a, a, 1 << 40, None) == mw.MOE_W4_ERR_UNSUPPORTED
    assert mw.moe_w4_forward_decode(p, 0, a, a, a, 1 << 40, None) == mw.MOE_W4_OK      # empty batch: no work
    assert mw.moe_w4_forward_prefill(p, 0, a, a, a, 1 << 40, None) == mw.MOE_W4_OK
    z = [a] * 6
    assert mw.moe_w4_route(p, 4, a, *z, None, a, 1 << 40, None) == mw.MOE_W4_ERR_INVALID   # inv missing
    assert mw.moe_w4_route(p, 4, a, *z, a, None, 1 << 40, None) == mw.MOE_W4_ERR_WORKSPACE
    L.gate = mw.MoeW4Mat(a + 4, a, a)
    assert mw.moe_w4_forward_prefill(p, 4, a, a, a, 1 << 40, None) == mw.MOE_W4_ERR_ALIGN
    L.gate = mw.MoeW4Mat(None, a, a)
    assert mw.moe_w4_forward_prefill(p, 4, a, a, a, 1 << 40, None) == mw.MOE_W4_ERR_INVALID


def test_strerror(mw):
    for code in (0, -1, -2, -3, -4, -5, -6, 42):
        assert isinstance(mw.moe_w4_strerror(code), str) and mw.moe_w4_strerror(code)


def test_router_prep_host_checks(mw):
    """The prepared router weights: size, and the host-side refusals (no device work)."""
    L = _layer(mw)
    n = mw.moe_w4_router_prep_bytes(ctypes.byref(L))
    assert n == 256 * 3 * 2048 * 2            # [ceil(E/128)*128][3H] bf16
    L2 = _layer(mw, E=200)
    assert mw.moe_w4_router_prep_bytes(ctypes.byref(L2)) == 256 * 3 * 2048 * 2
    assert mw.moe_w4_router_prep_bytes(None) == 0
    dst = 1 << 20
    assert mw.moe_w4_prepare_router(ctypes.byref(L), dst, n - 16, None) == mw.MOE_W4_ERR_WORKSPACE
    assert mw.moe_w4_prepare_router(ctypes.byref(L), dst + 8, n, None) == mw.MOE_W4_ERR_ALIGN
    assert mw.moe_w4_prepare_router(ctypes.byref(L), None, n, None) == mw.MOE_W4_ERR_INVALID
    L.router_prep = dst + 4                   # a misaligned prepared copy is refused by every call
    ws = 1 << 12
    assert mw.moe_w4_forward_prefill(ctypes.byref(L), 4, ws, ws, ws, 1 << 40, None) == mw.MOE_W4_ERR_ALIGN


def test_tile_override_values(mw):
    for bn, du in [(32, 1), (64, 2), (128, 4), (0, 0)]:
        assert mw.moe_w4_set_tile_override(bn, du) == mw.MOE_W4_OK
    for bn, du in [(16, 0), (96, 0), (256, 0), (0, 3), (0, 8), (-1, 0)]:
        assert mw.moe_w4_set_tile_override(bn, du) == mw.MOE_W4_ERR_INVALID
    assert mw.moe_w4_set_tile_override(0, 0) == mw.MOE_W4_OK


def test_ablation_mode_checked(mw):
    L = _layer(mw)
    ws = 1 << 12
    f = mw.moe_w4_ablation_prefill
    assert f(ctypes.byref(L), 4, ws, ws, ws, 1 << 40, 7, None, 0, None) == mw.MOE_W4_ERR_INVALID
    assert f(ctypes.byref(L), 0, ws, ws, ws, 1 << 40, mw.MOE_W4_ABLATE_HOST_ROUTING, None, 0, None) == mw.MOE_W4_OK
    # the separate dequantisation pass needs a scratch for every weight in fp16
    n = mw.moe_w4_ablation_scratch_bytes(ctypes.byref(L), mw.MOE_W4_ABLATE_SEPARATE_DEQUANT)
    assert n == 3 * 257 * 512 * 2048 * 2
    assert mw.moe_w4_ablation_scratch_bytes(ctypes.byref(L), mw.MOE_W4_ABLATE_HOST_ROUTING) == 0
    sep = mw.MOE_W4_ABLATE_SEPARATE_DEQUANT
    assert f(ctypes.byref(L), 4, ws, ws, ws, 1 << 40, sep, None, n, None) == mw.MOE_W4_ERR_INVALID
    assert f(ctypes.byref(L), 4, ws, ws, ws, 1 << 40, sep, ws + 8, n, None) == mw.MOE_W4_ERR_ALIGN
    assert f(ctypes.byref(L), 4, ws, ws, ws, 1 << 40, sep, ws, n - 16, None) == mw.MOE_W4_ERR_WORKSPACE
