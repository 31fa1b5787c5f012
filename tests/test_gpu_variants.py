"""GPU: the prefill's optional variants give the product path's results.

- the router weights prepared once per layer (moe_w4_prepare_router) against
  the split made in the workspace on every call: the same scores, so the
  same bits out;
- tile overrides (moe_w4_set_tile_override: token rows per block, row blocks
  per down unit): every choice against the oracle, and against the default
  tiles bit for bit (a tile changes which rows share an MMA, not the
  arithmetic of any output element);
- the measurement-only variants of moe_w4_ablation_prefill: the
  host-synchronised grouping (identical records) and the separate fp16
  dequantisation pass (identical fp16 weights in the same K order): identical
  bits out.
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


@pytest.fixture(scope="module")
def case(env):
    torch, mw = env
    L, x = S.draw_config("prefill_T512")
    return L, x, mw.DeviceLayer(L), O.moe_layer(L, x)["out"]


def test_router_prep_same_bits(env, case):
    torch, mw = env
    L, x, dl, ref = case
    assert dl.c.router_prep                      # prepared at construction
    plain = mw.DeviceLayer(L, prepare_router=False)
    assert not plain.c.router_prep
    xd = mw.tokens_to_device(x)
    a = _bits(torch, mw.forward_prefill(dl, xd))
    b = _bits(torch, mw.forward_prefill(plain, xd))
    torch.cuda.synchronize()
    assert np.array_equal(a, b)
    assert TOL.within(TOL.metrics(O.bf16_to_f64(a), ref))
    ra, rb = mw.route(dl, xd), mw.route(plain, xd)
    torch.cuda.synchronize()
    for k in ra:
        assert torch.equal(ra[k], rb[k]), k
    assert dl.status() == 0 and plain.status() == 0


@pytest.mark.parametrize("bn,du", [(32, 1), (64, 1), (64, 2), (64, 4), (128, 1), (128, 2)])
def test_tile_override(env, case, bn, du):
    torch, mw = env
    L, x, dl, ref = case
    xd = mw.tokens_to_device(x)
    base = _bits(torch, mw.forward_prefill(dl, xd))
    try:
        assert mw.moe_w4_set_tile_override(bn, du) == mw.MOE_W4_OK
        got = _bits(torch, mw.forward_prefill(dl, xd))
        torch.cuda.synchronize()
    finally:
        mw.moe_w4_set_tile_override(0, 0)
    assert TOL.within(TOL.metrics(O.bf16_to_f64(got), ref))
    assert np.array_equal(got, base)
    assert dl.status() == 0


@pytest.mark.parametrize("name", ["tiny_T4", "prefill_T512"])
def test_host_routing_ablation_same_bits(env, name):
    torch, mw = env
    L, x = S.draw_config(name)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    T = x.shape[0]
    ref_bits = _bits(torch, mw.forward_prefill(dl, xd))
    ws = dl.workspace(T)
    out = torch.full((T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    r = mw.moe_w4_ablation_prefill(ctypes.byref(dl.c), T, xd.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                   mw.MOE_W4_ABLATE_HOST_ROUTING, None, 0, st)
    assert r == mw.MOE_W4_OK
    torch.cuda.synchronize()
    assert np.array_equal(_bits(torch, out), ref_bits)
    assert dl.status() == 0


@pytest.mark.parametrize("name,bits,fmt", [("tiny_T4", 4, 0), ("prefill_T512", 4, 0), ("w8", 8, 0), ("w8", 8, 1)])
def test_separate_dequant_ablation_same_bits(env, name, bits, fmt):
    """Weights rebuilt in fp16 by a separate pass and read back by the GEMMs
    from shared memory: the same fp16 weights in the same K order as the fused
    dequantisers put in tensor memory, so the same bits out."""
    torch, mw = env
    if name == "w8":   # one-byte codes: a smaller layer (several tiles, ragged expert blocks)
        L = S.draw_layer(512, 64, 256, 4, 1.0, seed=31, bits=bits, fmt=fmt)
        x = S.draw_tokens(L, 200, 31)
    else:
        L, x = S.draw_config(name)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    T = x.shape[0]
    ref_bits = _bits(torch, mw.forward_prefill(dl, xd))
    ws = dl.workspace(T)
    mode = mw.MOE_W4_ABLATE_SEPARATE_DEQUANT
    n = mw.moe_w4_ablation_scratch_bytes(ctypes.byref(dl.c), mode)
    scratch = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.full((T, L.H), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    r = mw.moe_w4_ablation_prefill(ctypes.byref(dl.c), T, xd.data_ptr(), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                   mode, scratch.data_ptr(), n, st)
    assert r == mw.MOE_W4_OK
    torch.cuda.synchronize()
    assert np.array_equal(_bits(torch, out), ref_bits)
    assert dl.status() == 0


@pytest.mark.parametrize("name,bn", [("tiny_T4", 0), ("prefill_T512", 0), ("prefill_T512", 64),
                                     ("prefill_T4096", 0)])
def test_block_records_match_oracle_block_map(env, name, bn):
    """The GPU's block list against the oracle's block map: routed experts'
    blocks (expert, first row) exactly as oracle.block_map lists them for the
    block height in use, each with rows min(bn, count - first row) and first
    grouped position offsets[e] + first row; then the shared expert's blocks
    over all T tokens at positions T*k + first row."""
    torch, mw = env
    L, x = S.draw_config(name)
    dl = mw.DeviceLayer(L)
    T = x.shape[0]
    xd = mw.tokens_to_device(x)
    ws = dl.workspace(T)
    try:
        assert mw.moe_w4_set_tile_override(bn, 0) == mw.MOE_W4_OK
        mw.forward_prefill(dl, xd, ws=ws)
        n = mw.moe_w4_test_block_records_bytes(ctypes.byref(dl.c), T)
        rec = torch.zeros(n // 4, dtype=torch.int32, device="cuda")
        st = torch.cuda.current_stream().cuda_stream
        assert mw.moe_w4_test_block_records(ctypes.byref(dl.c), T, ws.data_ptr(), ws.numel(), rec.data_ptr(), n,
                                            st) == mw.MOE_W4_OK
        torch.cuda.synchronize()
    finally:
        mw.moe_w4_set_tile_override(0, 0)
    rec = rec.cpu().numpy()
    B = bn or 128
    nblk = int(rec[0]) // (L.I // 128)
    blocks = rec[2:2 + 4 * nblk].reshape(nblk, 4)
    idx, _, _, _ = O.route(O.bf16_to_f64(x), L.router_w, L.router_bias, L.shared_gate, L.top_k)
    counts, offsets, _, _ = O.group(idx, L.E)
    routed = blocks[blocks[:, 0] < L.E]
    assert [(int(e), int(r)) for e, r, _, _ in routed] == [(int(e), int(r)) for e, r in O.block_map(counts, B)]
    for e, r0, rows, p0 in routed:
        assert rows == min(B, counts[e] - r0) and p0 == offsets[e] + r0
    shared = blocks[blocks[:, 0] == L.E]
    assert [int(r) for r in shared[:, 1]] == list(range(0, T, B))
    for _, r0, rows, p0 in shared:
        assert rows == min(B, T - r0) and p0 == T * L.top_k + r0
    assert len(routed) + len(shared) == nblk


@pytest.mark.parametrize("E,T", [(18, 300), (36, 777), (256, 4096 + 130)])
def test_grouping_ragged_shapes(env, E, T):
    """The one-launch grouping on shapes the configs do not cover: an expert
    count that is not a multiple of 4 (scalar histogram reads), an odd number
    of token chunks with a ragged last one: routing and grouping bit-exact
    against the oracle, and the prefill within the layer tolerance."""
    torch, mw = env
    H, I, k = (256, 128, 2) if E < 64 else (2048, 512, 8)
    L = S.draw_layer(H, E, I, k, 1.0, seed=61 + E)
    x = S.draw_tokens(L, T, 61 + E)
    dl = mw.DeviceLayer(L)
    xd = mw.tokens_to_device(x)
    r = mw.route(dl, xd)
    torch.cuda.synchronize()
    idx, w, gam, _ = O.route(O.bf16_to_f64(x), L.router_w, L.router_bias, L.shared_gate, L.top_k)
    counts, offsets, perm, inv = O.group(idx, L.E)
    g = {kk: v.cpu().numpy() for kk, v in r.items()}
    assert np.array_equal(g["topk_idx"], idx)
    assert np.array_equal(g["counts"], counts) and np.array_equal(g["offsets"], offsets)
    assert np.array_equal(g["perm"], perm) and np.array_equal(g["inv"], inv)
    if E < 64:   # the oracle's layer is quick at this size
        out = _bits(torch, mw.forward_prefill(dl, xd))
        torch.cuda.synchronize()
        assert TOL.within(TOL.metrics(O.bf16_to_f64(out), O.moe_layer(L, x)["out"]))
    assert dl.status() == 0
