"""The allocation-free decode entry point against the regular one.

moe_w4_forward_decode_noalloc exists for callers that cannot allocate device
memory where they run the layer (an engine plugin whose host owns all device
memory, a real-time loop that must not wait on an allocator).  It takes no
workspace: its scratch is a fixed array inside the library.  This test calls it
through the C ABI twice in a row and checks each output against
moe_w4_forward_decode's (which uses a caller-owned workspace) within the layer
tolerance used everywhere else.  The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
from bit_quantized_sparse_gb300 import synthetic as S
from tests import tolerance as TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_quantized_sparse_gb300 import _build
    _build.build()
    from bit_quantized_sparse_gb300 import moe_w4 as mw
    return torch, mw


def _bits(torch, t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("name,T", [("decode_T1", None), ("decode_T1", 16), ("tiny_T4", None)])
def test_noalloc_matches_workspace_decode(env, name, T):
    torch, mw = env
    L, x = S.draw_config(name, T=T)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    n = x.shape[0]
    ref = _bits(torch, mw.forward_decode(dl, xd).clone())
    lib = ctypes.CDLL(mw.LIB_PATH)
    fn = lib.moe_w4_forward_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(mw.MoeW4Layer), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):                  # two calls in a row share the same scratch array
        out = torch.full((n, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert fn(ctypes.byref(dl.c), n, xd.data_ptr(), out.data_ptr(), stream) == mw.MOE_W4_OK
        torch.cuda.synchronize()
        got = _bits(torch, out)
        m = TOL.metrics(O.bf16_to_f64(got), O.bf16_to_f64(ref))
        assert TOL.within(m), (call, m)


def test_noalloc_rejects_oversized_calls(env):
    """A layer whose decode scratch exceeds the fixed array is refused cleanly."""
    torch, mw = env
    c = mw.MoeW4Layer()
    c.H, c.E, c.I, c.top_k = 4096, 1024, 4096, 8
    p = 1 << 12
    c.router_w = c.shared_gate = p
    for nm in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        setattr(c, nm, mw.MoeW4Mat(p, p, p))
    lib = ctypes.CDLL(mw.LIB_PATH)
    fn = lib.moe_w4_forward_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(mw.MoeW4Layer), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert fn(ctypes.byref(c), 16, p, p, None) == mw.MOE_W4_ERR_SCRATCH
    assert "scratch" in mw.moe_w4_strerror(mw.MOE_W4_ERR_SCRATCH)
