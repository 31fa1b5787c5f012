"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.

Bar: routing and grouping bit-exact (selected experts and their order,
per-expert counts, offsets, perm, inv); routing weights and the shared gate
within 1e-5; bf16 layer output within max|err| <= 2e-2 * rms(ref) and relative
L2 error <= 5e-3 against the float64 oracle.
"""
import numpy as np
import pytest

import oracle as O
from bit_quantized_sparse_gb300 import synthetic as S
from tests import tolerance as TOL

pytestmark = pytest.mark.gpu

W_TOL = 1e-5        # routing weights and shared gate


@pytest.fixture(scope="module")
def torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def mw(torch):
    from bit_quantized_sparse_gb300 import _build
    _build.build()
    from bit_quantized_sparse_gb300 import moe_w4
    return moe_w4


_CACHE = {}


def layer_of(mw, name, T=None):
    key = (name, T)
    if key not in _CACHE:
        L, x = S.draw_config(name, T=T)
        _CACHE[key] = (L, x, mw.DeviceLayer(L))
    return _CACHE[key]


def to_np_bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_out(got_bits, ref):
    """bf16 output against the float64 oracle (bar and its reading: tests/tolerance.py)."""
    got = O.bf16_to_f64(got_bits)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got))
    m = TOL.metrics(got, ref)
    assert TOL.within(m), m
    return m


def check_route(dev, L, x_bits):
    xf = O.bf16_to_f64(x_bits)
    idx, w, gam, _ = O.route(xf, L.router_w, L.router_bias, L.shared_gate, L.top_k)
    counts, offsets, perm, inv = O.group(idx, L.E)
    g = {k: v.cpu().numpy() for k, v in dev.items()}
    assert np.array_equal(g["topk_idx"], idx)
    assert np.max(np.abs(g["topk_w"] - w)) <= W_TOL
    assert np.max(np.abs(g["gamma"] - gam)) <= W_TOL
    assert np.array_equal(g["counts"], counts)
    assert np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["perm"], perm)
    assert np.array_equal(g["inv"], inv)


# ---------------------------------------------------------------------------
# routing and grouping: bit-exact at every configured size
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,T", [("tiny_T4", None), ("decode_T1", None), ("prefill_T512", None),
                                    ("prefill_T4096", None), ("long_T16384", 4096)])
def test_route_bit_exact(mw, torch, name, T):
    L, x, dl = layer_of(mw, name, T)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    check_route(r, L, x)
    assert dl.status() == 0


# ---------------------------------------------------------------------------
# prefill: grouped tensor-core path
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny_T4", "prefill_T512"])
def test_prefill_full(mw, torch, name):
    L, x, dl = layer_of(mw, name)
    out = mw.forward_prefill(dl, mw.tokens_to_device(x))
    torch.cuda.synchronize()
    ref = O.moe_layer(L, x)["out"]
    check_out(to_np_bits(out), ref)
    assert dl.status() == 0


def _sample(T, n, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=n, replace=False)]))


def test_prefill_T4096_every_row(mw, torch):
    """The 4K prefill (Zipf(1.0) routing): all 4096 rows against the oracle,
    element by element."""
    L, x, dl = layer_of(mw, "prefill_T4096")
    out = to_np_bits(mw.forward_prefill(dl, mw.tokens_to_device(x)))
    check_out(out, O.moe_layer(L, x)["out"])
    assert dl.status() == 0


def test_long_prompt_every_row(mw, torch):
    """The long prompt ("Optimizing on-device inference for Apple Silicon",
    section "Bound scratch with prompt chunking": chunking bounds the scratch
    and leaves the output unchanged).  Zipf(1.2) routing, 16384 rows as four
    4096-row calls sharing one workspace: every row of every chunk against the
    oracle; one 16384-row call gives the same bytes; then the 64 batch-1 decode
    rows on the same layer (the one-kernel path), each against the oracle."""
    c = S.CONFIGS["long_T16384"]
    L, x, dl = layer_of(mw, "long_T16384")
    T, chunk = c["T"], c["chunk"]
    assert x.shape[0] == T
    xd = mw.tokens_to_device(x)
    n = dl.workspace_size(chunk)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    mw._check(mw.moe_w4_workspace_init(ws.data_ptr(), n, torch.cuda.current_stream().cuda_stream), "init")
    parts = [mw.forward_prefill(dl, xd[i:i + chunk], ws=ws).clone() for i in range(0, T, chunk)]
    whole = mw.forward_prefill(dl, xd)
    torch.cuda.synchronize()
    st = int(ws[mw.moe_w4_status_offset():][:4].view(torch.int32).item())
    assert st == 0 and dl.status() == 0
    chunked = torch.cat(parts)
    assert torch.equal(whole.view(torch.int16), chunked.view(torch.int16))
    ref = O.moe_layer(L, x)["out"]
    got = to_np_bits(chunked)
    for i in range(0, T, chunk):
        check_out(got[i:i + chunk], ref[i:i + chunk])
    # 64 consecutive batch-1 decode steps, fresh seeded rows (no model feedback)
    xdec = S.draw_tokens(L, c["decode_steps"], c["seed"], stream=1)
    outs = [mw.forward_decode(dl, mw.tokens_to_device(xdec[i:i + 1])).clone() for i in range(xdec.shape[0])]
    torch.cuda.synchronize()
    got_dec = np.concatenate([to_np_bits(o) for o in outs])
    ref_dec = O.moe_layer(L, xdec)["out"]
    for i in range(xdec.shape[0]):
        check_out(got_dec[i:i + 1], ref_dec[i:i + 1])
    _, nk = _traced_decode(mw, torch, dl, xdec[:1])
    assert nk == 1, nk                      # the one-kernel batch-1 decode ran
    assert dl.status() == 0


@pytest.mark.parametrize("name", ["w8_T512", "e4m3_T512"])
def test_byte_codes_prefill_sampled(mw, torch, name):
    """The one-byte-code layers at the benchmark's chunk size (4096 rows, the
    size the format-variant measurement times): routing bit-exact, sampled
    rows against the oracle."""
    L, x, dl = layer_of(mw, name, 4096)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    check_route(r, L, x)
    out = to_np_bits(mw.forward_prefill(dl, xd))
    rows = _sample(x.shape[0], 32, 11)
    check_out(out[rows], O.moe_layer(L, x, tokens=rows)["out"])
    assert dl.status() == 0


def test_prefill_single_token_and_ragged(mw, torch):
    L, x, dl = layer_of(mw, "prefill_T512")
    for T in (1, 3, 129, 333):
        out = to_np_bits(mw.forward_prefill(dl, mw.tokens_to_device(x[:T])))
        rows = _sample(T, min(T, 8), T)
        check_out(out[rows], O.moe_layer(L, x[:T], tokens=rows)["out"])


def test_prefill_chunked_equals_unchunked(mw, torch):
    L, x, dl = layer_of(mw, "prefill_T4096")
    xd = mw.tokens_to_device(x[:2048])
    whole = mw.forward_prefill(dl, xd).clone()
    parts = torch.cat([mw.forward_prefill(dl, xd[i:i + 512]).clone() for i in range(0, 2048, 512)])
    torch.cuda.synchronize()
    assert torch.equal(whole.view(torch.int16), parts.view(torch.int16))


def test_prefill_deterministic(mw, torch):
    L, x, dl = layer_of(mw, "prefill_T512")
    xd = mw.tokens_to_device(x)
    a = mw.forward_prefill(dl, xd).clone()
    b = mw.forward_prefill(dl, xd).clone()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_prefill_all_tokens_to_same_experts(mw, torch):
    """Degenerate routing: a router bias makes every token pick experts 0..7,
    so eight groups hold all T rows and the rest are empty."""
    L, _, _ = layer_of(mw, "prefill_T512")
    import copy
    L2 = copy.copy(L)
    bias = np.full(L.E, -50.0, np.float32)
    bias[:L.top_k] = 5.0 * np.arange(L.top_k, 0, -1)
    L2.router_bias = bias
    x = S.draw_tokens(L2, 300, seed=11)
    dl = mw.DeviceLayer(L2)
    r = mw.route(dl, mw.tokens_to_device(x))
    out = to_np_bits(mw.forward_prefill(dl, mw.tokens_to_device(x)))
    torch.cuda.synchronize()
    check_route(r, L2, x)
    assert np.all(r["counts"].cpu().numpy()[:L.top_k] == 300) and r["counts"].cpu().numpy()[L.top_k:].sum() == 0
    rows = _sample(300, 12, 3)
    check_out(out[rows], O.moe_layer(L2, x, tokens=rows)["out"])


def test_small_layer_top1(mw, torch):
    """E = 16, top_k = 1: every routing weight is exactly 1."""
    L = S.draw_layer(256, 16, 128, 1, None, seed=21)
    x = S.draw_tokens(L, 64, seed=21)
    dl = mw.DeviceLayer(L)
    r = mw.route(dl, mw.tokens_to_device(x))
    torch.cuda.synchronize()
    check_route(r, L, x)
    assert np.all(r["topk_w"].cpu().numpy() == 1.0)
    ref = O.moe_layer(L, x)["out"]
    check_out(to_np_bits(mw.forward_prefill(dl, mw.tokens_to_device(x))), ref)
    check_out(to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[:16]))), ref[:16])


def test_widths_not_multiple_of_256(mw, torch):
    """H = I = 384: multiples of 128 (the supported granularity) but not of 256,
    so rows of x and h end inside a 256-column block and the quantisation groups
    per row (6) are not a multiple of 8.  Routing, prefill and decode against the
    oracle."""
    L = S.draw_layer(384, 32, 384, 4, 1.0, seed=31)
    x = S.draw_tokens(L, 200, seed=31)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    check_route(r, L, x)
    ref = O.moe_layer(L, x)["out"]
    check_out(to_np_bits(mw.forward_prefill(dl, xd)), ref)
    check_out(to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[:3]))), ref[:3])
    check_out(to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[7:8]))), ref[7:8])
    assert dl.status() == 0


@pytest.mark.parametrize("H,E,I,k", [(1024, 128, 256, 4), (2048, 64, 1024, 4)])
def test_other_shapes(mw, torch, H, E, I, k):
    """Shapes off the benchmark's.  (1024, 128, 256, 4): the one-kernel T=1
    decode with shapes taken at run time.  (2048, 64, 1024, 4): a down
    projection whose K (I = 1024) exceeds the tensor-memory A ring, so every
    down unit is one row block; E = 64 sends T=1 decode to the grouped path.
    Routing, prefill and decode (1 and 5 rows) against the oracle."""
    L = S.draw_layer(H, E, I, k, 1.0, seed=40 + k)
    x = S.draw_tokens(L, 96, seed=41)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    check_route(r, L, x)
    ref = O.moe_layer(L, x)["out"]
    check_out(to_np_bits(mw.forward_prefill(dl, xd)), ref)
    for a, b in ((0, 1), (5, 6), (10, 15)):
        check_out(to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[a:b]))), ref[a:b])
    assert dl.status() == 0


def _traced_decode(mw, torch, dl, x_rows):
    """One decode call with the library's kernel timing events set: the output
    (bf16 bits) and the number of kernels the call launched."""
    import ctypes
    n = 12
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
    mw._check(mw.moe_w4_set_trace_events(arr, n), "trace")
    try:
        out = mw.forward_decode(dl, mw.tokens_to_device(x_rows))
        torch.cuda.synchronize()
        nk = mw.moe_w4_last_traced_kernels()
    finally:
        mw.moe_w4_set_trace_events(None, 0)
    return to_np_bits(out), nk


@pytest.mark.parametrize("name", ["w8_tiny_T4", "w8_T512", "e4m3_tiny_T4", "e4m3_T512"])
def test_w8_layer(mw, torch, name):
    """The one-byte weight-format variants (four codes per word; unsigned
    8-bit affine codes or FP8 E4M3 codes): routing, prefill and decode (1 and 4
    rows: the one-kernel path, once per row, for the full-size layer; the
    grouped path for the tiny one) against the oracle; the allocation-free
    decode runs the one-kernel path for the full-size layer at T = 1 and 4 and
    declines the tiny layer, whose fallback kernels unpack nibbles."""
    import ctypes
    L, x = S.draw_config(name)
    assert L.code_bits == 8
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    check_route(r, L, x)
    ref = O.moe_layer(L, x)["out"]
    check_out(to_np_bits(mw.forward_prefill(dl, xd)), ref)
    out1, nk = _traced_decode(mw, torch, dl, x[:1])
    check_out(out1, ref[:1])
    # the full-size layer takes the one-kernel batch-1 decode, the tiny one the grouped path
    assert nk == (1 if L.H == 2048 else 7), nk   # grouped path: router, top-k, grouping, gather, 2 GEMMs, combine
    if x.shape[0] >= 8:
        check_out(to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[4:8]))), ref[4:8])
    # the allocation-free decode: the one-kernel path, once per row (full-size
    # layer only); its fallback kernels unpack nibbles, so the tiny layer's
    # one-byte codes are declined
    out = torch.empty((4, L.H), dtype=torch.bfloat16, device="cuda")
    for T in (1, 4):
        if x.shape[0] < T:
            continue
        rc = mw.moe_w4_forward_decode_noalloc(ctypes.byref(dl.c), T, xd.data_ptr(), out.data_ptr(), None)
        if L.H == 2048:
            assert rc == mw.MOE_W4_OK
            torch.cuda.synchronize()
            check_out(to_np_bits(out[:T]), ref[:T])
        else:
            assert rc == mw.MOE_W4_ERR_UNSUPPORTED
    assert dl.status() == 0


# ---------------------------------------------------------------------------
# decode: fused GEMV path
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,T", [("decode_T1", None), ("tiny_T4", None), ("decode_T1", 16)])
def test_decode(mw, torch, name, T):
    L, x, dl = layer_of(mw, name, T)
    out = mw.forward_decode(dl, mw.tokens_to_device(x))
    torch.cuda.synchronize()
    check_out(to_np_bits(out), O.moe_layer(L, x)["out"])
    assert dl.status() == 0


@pytest.mark.parametrize("name", ["decode_T1", "prefill_T512"])
def test_decode_single_tokens(mw, torch, name):
    """Batch-1 decode (the one-kernel path for these shapes) on 12 tokens, one
    call each, uniform and Zipf-skewed routing, against the oracle."""
    L, x, dl = layer_of(mw, name)
    xs = S.draw_tokens(L, 12, seed=99, stream=5)
    outs = []
    for t in range(12):
        outs.append(mw.forward_decode(dl, mw.tokens_to_device(xs[t:t + 1])).clone())
    torch.cuda.synchronize()
    got = np.concatenate([to_np_bits(o) for o in outs])
    check_out(got, O.moe_layer(L, xs)["out"])
    assert dl.status() == 0


@pytest.mark.parametrize("T", [2, 3, 5])
def test_decode_rows_fused(mw, torch, T):
    """Decode calls of a few rows run the one-kernel batch-1 decode once per
    row: moe_w4_decode_path says so, the trace counts T kernels, and the output
    equals the rows' separate batch-1 calls bit for bit and the oracle within
    the layer tolerance.  With the row limit set to 1 the same call takes the
    grouped path (7 kernels), also within the tolerance; 6 rows take it by
    default."""
    L, x, dl = layer_of(mw, "decode_T1", 16)
    ref = O.moe_layer(L, x[:T])["out"]
    assert mw.decode_path(dl, T) == mw.MOE_W4_PATH_FUSED_ROWS
    assert mw.decode_path(dl, 6) == mw.MOE_W4_PATH_GROUPED
    rows, nk = _traced_decode(mw, torch, dl, x[:T])
    assert nk == T, nk
    check_out(rows, ref)
    singles = np.concatenate([to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[t:t + 1])))
                              for t in range(T)])
    assert np.array_equal(rows, singles)
    assert mw.moe_w4_set_decode_fused_rows(1) == mw.MOE_W4_OK
    try:
        assert mw.decode_path(dl, T) == mw.MOE_W4_PATH_GROUPED
        grouped, nk = _traced_decode(mw, torch, dl, x[:T])
    finally:
        assert mw.moe_w4_set_decode_fused_rows(0) == mw.MOE_W4_OK
    assert nk == 7, nk   # router, top-k, grouping, gather, 2 GEMMs, combine
    check_out(grouped, ref)
    assert mw.decode_path(dl, T) == mw.MOE_W4_PATH_FUSED_ROWS
    assert dl.status() == 0


@pytest.mark.parametrize("allow", [0, 1])
def test_decode_refused_launch_falls_back(mw, torch, allow):
    """A refused cooperative launch of the one-kernel decode (simulated on the
    host by moe_w4_test_refuse_fused_after: nothing is refused for real) sends
    the rows not yet enqueued to the grouped path: a 3-row call with 0 or 1 rows
    allowed on the one-kernel path ends on the grouped path's 7 kernels and
    matches the oracle with a clear status."""
    L, x, dl = layer_of(mw, "decode_T1", 16)
    ref = O.moe_layer(L, x[:3])["out"]
    assert mw.moe_w4_test_refuse_fused_after(allow) == mw.MOE_W4_OK
    try:
        got, nk = _traced_decode(mw, torch, dl, x[:3])
    finally:
        mw.moe_w4_test_refuse_fused_after(-1)
    assert nk == 7, nk
    check_out(got, ref)
    assert dl.status() == 0


def test_decode_matches_prefill(mw, torch):
    L, x, dl = layer_of(mw, "decode_T1", 16)
    xd = mw.tokens_to_device(x)
    a = O.bf16_to_f64(to_np_bits(mw.forward_decode(dl, xd)))
    b = to_np_bits(mw.forward_prefill(dl, xd))
    check_out(b, a)


def test_decode_repeated_calls(mw, torch):
    """The decode router's completion counter is reset by the last CTA, so
    back-to-back calls give identical results."""
    L, x, dl = layer_of(mw, "decode_T1")
    xd = mw.tokens_to_device(x)
    outs = [mw.forward_decode(dl, xd).clone() for _ in range(5)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert dl.status() == 0


def test_gpu_workspace_errors(mw, torch):
    import ctypes
    L, x, dl = layer_of(mw, "tiny_T4")
    xd = mw.tokens_to_device(x)
    out = torch.empty((4, L.H), dtype=torch.bfloat16, device="cuda")
    need = dl.workspace_size(4)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert mw.moe_w4_forward_prefill(ctypes.byref(dl.c), 4, xd.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                     need - 1, st) == mw.MOE_W4_ERR_WORKSPACE
    assert mw.moe_w4_forward_prefill(ctypes.byref(dl.c), 4, xd.data_ptr() + 2, out.data_ptr(), ws.data_ptr(),
                                     need, st) == mw.MOE_W4_ERR_ALIGN
    assert mw.moe_w4_forward_prefill(ctypes.byref(dl.c), 4, xd.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                     need, st) == mw.MOE_W4_OK
    torch.cuda.synchronize()


def test_prefill_fp16_range_status(mw, torch):
    """x within the fp16 range, but large enough that the weighted SwiGLU output
    is not: the prefill sets MOE_W4_STATUS_FP16_RANGE in the status word; a
    call on ordinary inputs leaves it clear."""
    L, x = S.draw_config("tiny_T4")
    dl = mw.DeviceLayer(L)
    mw.forward_prefill(dl, mw.tokens_to_device(x))
    torch.cuda.synchronize()
    assert dl.status() == 0
    xf = S.bf16_bits_to_f32(x).astype(np.float64)
    big = S.f32_to_bf16_bits((xf * (60000.0 / np.abs(xf).max())).astype(np.float32))
    mw.forward_prefill(dl, mw.tokens_to_device(big))
    torch.cuda.synchronize()
    assert dl.status() & mw.MOE_W4_STATUS_FP16_RANGE


def _scaled_layer(L, a):
    """The layer with every scale and bias times 2^a (exact in bf16) and the router
    and shared-gate weights times 2^a too: with activations times 2^-a the routing
    scores x . W_r and the shared gate are unchanged bit for bit."""
    import copy
    L2 = copy.deepcopy(L)
    for nm in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down"):
        m = getattr(L2, nm)
        for f in ("scales", "biases"):
            v = S.bf16_bits_to_f32(getattr(m, f)).astype(np.float64) * 2.0 ** a
            setattr(m, f, S.f32_to_bf16_bits(v.astype(np.float32)))
    L2.router_w = (L.router_w.astype(np.float64) * 2.0 ** a).astype(np.float32)
    L2.shared_gate = (L.shared_gate.astype(np.float64) * 2.0 ** a).astype(np.float32)
    return L2


def test_large_scales_small_activations(mw, torch):
    """Scales of 1e1 .. 4e2 (the generator's times 2^12, exact in bf16) with
    activations near 6e-5 (times 2^-14), router weights times 2^12 (the same
    scores): the rebuilt weights, h and the expert outputs (up to about 4e4) stay
    within fp16, so prefill and a 4-row decode on the grouped path match the
    oracle and the status word stays clear.  (The one-kernel batch-1 decode, which
    by default also takes calls of up to 5 rows, holds half of x divided by 16 in
    fp16 with 4-bit codes, below the fp16 normal range at these activations: not
    run here.)"""
    L0 = S.draw_layer(2048, 256, 512, 8, 1.0, seed=57)
    x0 = S.draw_tokens(L0, 40, seed=57)
    L = _scaled_layer(L0, 12)
    x = S.f32_to_bf16_bits((S.bf16_bits_to_f32(x0).astype(np.float64) * 2.0 ** -14).astype(np.float32))
    assert 30 < np.median(S.bf16_bits_to_f32(L.gate.scales)) < 100
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    check_route(r, L, x)
    ref = O.moe_layer(L, x)["out"]
    check_out(to_np_bits(mw.forward_prefill(dl, xd)), ref)
    assert mw.moe_w4_set_decode_fused_rows(1) == mw.MOE_W4_OK
    try:
        got = to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x[3:7])))
    finally:
        assert mw.moe_w4_set_decode_fused_rows(0) == mw.MOE_W4_OK
    check_out(got, ref[3:7])
    assert dl.status() == 0


def test_weight_range_status(mw, torch):
    """One group whose rebuilt weights exceed the fp16 range (scale 2^13, so
    15 s > 65504) sets MOE_W4_STATUS_FP16_RANGE in the prefill; activations near
    zero keep every other fp16 value in range, so the bit comes from the weights."""
    L, _ = S.draw_config("tiny_T4")
    import copy
    L2 = copy.deepcopy(L)
    sc = L2.gate.scales.copy()
    sc[:, 0, 0] = S.f32_to_bf16_bits(np.array([8192.0], np.float32))[0]   # every expert's row 0, group 0
    L2.gate.scales = sc
    L2.sh_gate.scales = L2.sh_gate.scales.copy()
    L2.sh_gate.scales[0, 0] = sc[0, 0, 0]
    x = S.draw_tokens(L2, 4, seed=5)
    dl = mw.DeviceLayer(L2)
    mw.forward_prefill(dl, mw.tokens_to_device(x))
    torch.cuda.synchronize()
    assert dl.status() & mw.MOE_W4_STATUS_FP16_RANGE


def test_decode_wait_timeout_is_reported(mw, torch):
    """Failure detection without a GPU fault: with the test hook on, one cluster
    of the batch-1 kernel does not publish its router sums, so the other CTAs'
    bounded waits run out.  The call completes, the status word reports the
    timeout, the context stays usable, and after re-initialising the workspace
    the next call matches the oracle."""
    import ctypes
    L, x = S.draw_config("decode_T1")
    dl = mw.DeviceLayer(L)
    ws = dl.workspace(1)
    xd = mw.tokens_to_device(x)
    stream = torch.cuda.current_stream().cuda_stream
    mw._check(mw.moe_w4_test_skip_publish(ws.data_ptr(), ws.numel(), 1, stream), "hook")
    out = torch.empty((1, L.H), dtype=torch.bfloat16, device="cuda")
    mw._check(mw.moe_w4_forward_decode(ctypes.byref(dl.c), 1, xd.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                       ws.numel(), stream), "decode")
    torch.cuda.synchronize()   # returns: every wait is bounded
    assert dl.status() & mw.MOE_W4_STATUS_WAIT_TIMEOUT
    mw._check(mw.moe_w4_workspace_init(ws.data_ptr(), ws.numel(), stream), "init")
    torch.cuda.synchronize()
    assert dl.status() == 0
    check_out(to_np_bits(mw.forward_decode(dl, xd)), O.moe_layer(L, x)["out"])
    assert dl.status() == 0


def test_decode_after_timeout_without_reinit(mw, torch):
    """A batch-1 call that gives up its waits still advances the call counter
    its exchanged words are tagged with: with the test hook turned off again and
    no workspace re-initialisation, the next call must not take any of the
    aborted call's words for its own, so it matches the oracle (the sticky
    status word keeps the earlier timeout bit)."""
    import ctypes
    L, x = S.draw_config("decode_T1")
    dl = mw.DeviceLayer(L)
    ws = dl.workspace(1)
    xd = mw.tokens_to_device(x)
    stream = torch.cuda.current_stream().cuda_stream
    mw.forward_decode(dl, xd)             # a normal call first: the counter is past 0
    mw._check(mw.moe_w4_test_skip_publish(ws.data_ptr(), ws.numel(), 1, stream), "hook")
    out = torch.empty((1, L.H), dtype=torch.bfloat16, device="cuda")
    mw._check(mw.moe_w4_forward_decode(ctypes.byref(dl.c), 1, xd.data_ptr(), out.data_ptr(), ws.data_ptr(),
                                       ws.numel(), stream), "decode")
    mw._check(mw.moe_w4_test_skip_publish(ws.data_ptr(), ws.numel(), 0, stream), "hook off")
    torch.cuda.synchronize()
    assert dl.status() & mw.MOE_W4_STATUS_WAIT_TIMEOUT
    x2 = S.draw_tokens(L, 3, seed=123)
    for t in range(3):
        got = to_np_bits(mw.forward_decode(dl, mw.tokens_to_device(x2[t:t + 1])))
        check_out(got, O.moe_layer(L, x2[t:t + 1])["out"])


def test_trace_events_outside_capture(mw, torch):
    """Kernel timing events recorded around an eager (not captured) call: the call
    succeeds and every event completes in order."""
    import ctypes
    L, x, dl = layer_of(mw, "tiny_T4")
    n = 10
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    arr = (ctypes.c_void_p * n)(*[e.cuda_event for e in evs])
    mw._check(mw.moe_w4_set_trace_events(arr, n), "trace")
    try:
        out = mw.forward_prefill(dl, mw.tokens_to_device(x))
        torch.cuda.synchronize()
        nk = mw.moe_w4_last_traced_kernels()
    finally:
        mw.moe_w4_set_trace_events(None, 0)
    assert nk == 7   # router, top-k, grouping, gather, 2 GEMMs, combine
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(nk)]
    assert all(t >= 0 for t in times)
    check_out(to_np_bits(out), O.moe_layer(L, x)["out"])
