"""The allocation-free decode entry point against the regular one.

moe_w4_forward_decode_noalloc exists for callers that cannot allocate device
memory where they run the layer (an engine plugin whose host owns all device
memory, a real-time loop that must not wait on an allocator).  It takes no
workspace: its scratch is a fixed array inside the library, shared by every
call.  These tests call it through the C ABI, two calls in a row, and check
each output against moe_w4_forward_decode's (which uses a caller-owned
workspace) and against the oracle, within the layer tolerance used everywhere
else; a sequence of calls that alternates batch sizes and layers checks that
one call's leftovers in the shared array never leak into the next, and that
the status word (read through moe_w4_noalloc_status) stays clear.  The file
name makes pytest collect it last.
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


def _fn(mw):
    lib = ctypes.CDLL(mw.LIB_PATH)
    fn = lib.moe_w4_forward_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(mw.MoeW4Layer), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fn


def _status(torch, mw):
    """The allocation-free path's status word, copied into device memory."""
    word = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert mw.moe_w4_noalloc_status(word.data_ptr(), torch.cuda.current_stream().cuda_stream) == mw.MOE_W4_OK
    torch.cuda.synchronize()
    return int(word.item())


@pytest.mark.parametrize("name,T", [("decode_T1", None), ("decode_T1", 16), ("tiny_T4", None)])
def test_noalloc_matches_workspace_decode(env, name, T):
    torch, mw = env
    L, x = S.draw_config(name, T=T)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    n = x.shape[0]
    ref = _bits(torch, mw.forward_decode(dl, xd).clone())
    oracle = O.moe_layer(L, x)["out"]
    fn = _fn(mw)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):                  # two calls in a row share the same scratch array
        out = torch.full((n, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert fn(ctypes.byref(dl.c), n, xd.data_ptr(), out.data_ptr(), stream) == mw.MOE_W4_OK
        torch.cuda.synchronize()
        got = O.bf16_to_f64(_bits(torch, out))
        m = TOL.metrics(got, O.bf16_to_f64(ref))
        assert TOL.within(m), (call, m)
        m = TOL.metrics(got, oracle)
        assert TOL.within(m), (call, "oracle", m)
        assert _status(torch, mw) == 0


def test_noalloc_alternating_sizes_and_layers(env):
    """T = 1, T = 16, T = 1 on the full-size layer, then a different full-size
    layer at T = 1 and the tiny layer at T = 4: the T >= 2 kernels write where
    nothing of the one-kernel T = 1 path lives, and the T = 1 path's exchange
    words carry call tags that never repeat, so every output matches the
    oracle and the status word stays clear."""
    torch, mw = env
    fn = _fn(mw)
    stream = torch.cuda.current_stream().cuda_stream
    La, xa = S.draw_config("decode_T1", T=16)
    Lb = S.draw_layer(2048, 256, 512, 8, 1.2, seed=77)
    xb = S.draw_tokens(Lb, 2, seed=77)
    Lt, xt = S.draw_config("tiny_T4")
    da, db, dt = mw.DeviceLayer(La), mw.DeviceLayer(Lb), mw.DeviceLayer(Lt)
    ref_a = O.moe_layer(La, xa)["out"]
    seq = [(da, xa[:1], ref_a[:1]), (da, xa, ref_a), (da, xa[5:6], ref_a[5:6]),
           (db, xb[:1], O.moe_layer(Lb, xb[:1])["out"]), (dt, xt, O.moe_layer(Lt, xt)["out"]),
           (da, xa[9:10], ref_a[9:10])]
    for i, (dl, x, ref) in enumerate(seq):
        n = x.shape[0]
        xd = mw.tokens_to_device(x)
        out = torch.full((n, dl.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert fn(ctypes.byref(dl.c), n, xd.data_ptr(), out.data_ptr(), stream) == mw.MOE_W4_OK
        torch.cuda.synchronize()
        m = TOL.metrics(O.bf16_to_f64(_bits(torch, out)), ref)
        assert TOL.within(m), (i, m)
        assert _status(torch, mw) == 0, i


def test_noalloc_rejects_oversized_calls(env):
    """A layer whose decode scratch exceeds the fixed array is refused cleanly."""
    torch, mw = env
    c = mw.MoeW4Layer()
    c.H, c.E, c.I, c.top_k = 4096, 1024, 4096, 8
    p = 1 << 12
    c.router_w = c.shared_gate = p
    for nm in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        setattr(c, nm, mw.MoeW4Mat(p, p, p))
    fn = _fn(mw)
    assert fn(ctypes.byref(c), 16, p, p, None) == mw.MOE_W4_ERR_SCRATCH
    assert "scratch" in mw.moe_w4_strerror(mw.MOE_W4_ERR_SCRATCH)


def test_noalloc_wait_timeout_then_valid_call(env):
    """Failure detection on the allocation-free path, without a fault: with the
    test hook on, one CTA of the batch-1 kernel skips publishing its router
    scores, the others' bounded waits run out (about 2 s) and the status word
    reports MOE_W4_STATUS_WAIT_TIMEOUT; the aborting CTAs advance the call
    counter, so the next call (hook off) is right with a clear status."""
    torch, mw = env
    fn = _fn(mw)
    stream = torch.cuda.current_stream().cuda_stream
    L, x = S.draw_config("decode_T1", T=2)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    ref = O.moe_layer(L, x)["out"]
    out = torch.full((1, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    try:
        assert mw.moe_w4_noalloc_test_skip_publish(1) == mw.MOE_W4_OK
        assert fn(ctypes.byref(dl.c), 1, xd[:1].data_ptr(), out.data_ptr(), stream) == mw.MOE_W4_OK
        torch.cuda.synchronize()
    finally:
        mw.moe_w4_noalloc_test_skip_publish(0)
    assert _status(torch, mw) & mw.MOE_W4_STATUS_WAIT_TIMEOUT
    for i in range(2):
        assert fn(ctypes.byref(dl.c), 1, xd[i:i + 1].data_ptr(), out.data_ptr(), stream) == mw.MOE_W4_OK
        torch.cuda.synchronize()
        m = TOL.metrics(O.bf16_to_f64(_bits(torch, out)), ref[i:i + 1])
        assert TOL.within(m), (i, m)
        assert _status(torch, mw) == 0, i


def test_noalloc_refused_launch_falls_back(env):
    """A refused cooperative launch of the one-kernel path in the allocation-free
    decode (simulated on the host by moe_w4_test_refuse_fused_after): with 1 of
    3 rows allowed, the other two take the CUDA-core kernels and the output
    matches the oracle with a clear status; one-byte codes, which those kernels
    cannot read, return MOE_W4_ERR_LAUNCH instead."""
    torch, mw = env
    fn = _fn(mw)
    stream = torch.cuda.current_stream().cuda_stream
    for name, ok in (("decode_T1", True), ("w8_T512", False)):
        L, x = S.draw_config(name, T=3)
        dl = mw.DeviceLayer(L)
        xd = mw.tokens_to_device(x)
        out = torch.full((3, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert mw.moe_w4_test_refuse_fused_after(1) == mw.MOE_W4_OK
        try:
            rc = fn(ctypes.byref(dl.c), 3, xd.data_ptr(), out.data_ptr(), stream)
            torch.cuda.synchronize()
        finally:
            mw.moe_w4_test_refuse_fused_after(-1)
        if ok:
            assert rc == mw.MOE_W4_OK
            m = TOL.metrics(O.bf16_to_f64(_bits(torch, out)), O.moe_layer(L, x)["out"])
            assert TOL.within(m), m
            assert _status(torch, mw) == 0
        else:
            assert rc == mw.MOE_W4_ERR_LAUNCH
