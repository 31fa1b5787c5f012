"""The debug build (libmoe_w4_debug.so: device-side bounds checks on every
index read from the routing records, MOE_W4_STATUS_BAD_INDEX and a clamped
access on a failed check).

CPU: it compiles for sm_103a and exports every entry point of the product
library.  GPU: on valid inputs the checks never fire and the outputs are the
product library's bit for bit (prefill, the one-kernel batch-1 decode and a
multi-row decode), with the status word clear.
"""
import ctypes
import os
import shutil

import numpy as np
import pytest

from bit_quantized_sparse_gb300 import synthetic as S


def _debug_lib():
    from bit_quantized_sparse_gb300 import _build
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    return _build.build(debug=True)


def test_debug_build_exports_the_abi():
    path = _debug_lib()
    from bit_quantized_sparse_gb300 import _build
    _build.build()
    from bit_quantized_sparse_gb300 import moe_w4 as mw
    lib = ctypes.CDLL(path)
    for name in mw.EXPORTED:
        assert hasattr(lib, name), name


def _bind(lib, mw):
    P = ctypes.POINTER(mw.MoeW4Layer)
    for name in ("moe_w4_forward_prefill", "moe_w4_forward_decode"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [P, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                      ctypes.c_void_p]
    lib.moe_w4_workspace_init.restype = ctypes.c_int
    lib.moe_w4_workspace_init.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    return lib


@pytest.mark.gpu
@pytest.mark.parametrize("name,T,fn", [("prefill_T512", None, "moe_w4_forward_prefill"),
                                       ("decode_T1", None, "moe_w4_forward_decode"),
                                       ("decode_T1", 4, "moe_w4_forward_decode"),
                                       ("tiny_T4", None, "moe_w4_forward_prefill")])
def test_debug_build_same_bits(name, T, fn):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = _debug_lib()
    from bit_quantized_sparse_gb300 import _build
    _build.build()
    from bit_quantized_sparse_gb300 import moe_w4 as mw
    dbg = _bind(ctypes.CDLL(path), mw)
    L, x = S.draw_config(name, T=T)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    n = x.shape[0]
    ref = (mw.forward_prefill if fn == "moe_w4_forward_prefill" else mw.forward_decode)(dl, xd)
    ws = torch.empty(dl.workspace_size(n), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert dbg.moe_w4_workspace_init(ws.data_ptr(), ws.numel(), st) == 0
    out = torch.full((n, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert getattr(dbg, fn)(ctypes.byref(dl.c), n, xd.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(), st) == 0
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(bits(out), bits(ref))
    off = mw.moe_w4_status_offset()
    assert int(ws[off:off + 4].view(torch.int32).item()) == 0
