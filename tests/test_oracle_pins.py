"""Pins for the CPU oracle: values fixed by the pages, closed forms, invariants,
library routines for special cases and brute force on tiny inputs.

Every check is a plain function raising AssertionError, so the planted-mistake
tests at the bottom can re-run it against a deliberately broken oracle and
demand that it fails.
"""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle.moe_w4_oracle as O
from bit_quantized_sparse_gb300 import synthetic as S
from tests import brute_force as BF

GOLD = os.path.join(os.path.dirname(__file__), "golden")
bf = S.f32_to_bf16_bits


def _lines(name):
    with open(os.path.join(GOLD, name)) as f:
        for ln in f:
            ln = ln.strip()
            if ln and not ln.startswith("#"):
                yield ln


# ---------------------------------------------------------------------------
# dequantisation
# ---------------------------------------------------------------------------
def check_dequant_golden():
    n = 0
    for ln in _lines("dequant_cases.txt"):
        tok = ln.split()
        word = np.array([[int(tok[0], 16)] * 8], dtype=np.uint32)      # one row, 64 columns
        s = bf(np.array([[float(tok[1])]], np.float32))
        b = bf(np.array([[float(tok[2])]], np.float32))
        want = np.array([float(v) for v in tok[3:11]])
        got = O.dequant(word, s, b)
        assert got.shape == (1, 64)
        assert np.array_equal(got[0, :8], want), (tok[0], got[0, :8], want)
        assert np.array_equal(got[0, 8:16], want)
        n += 1
    assert n == 7


def check_group_axis():
    """2 rows x 128 columns (two groups per row), every code 1: w = s + b of
    the group (row r, column c // 64)."""
    codes = np.full((2, 16), 0x11111111, dtype=np.uint32)
    s = bf(np.array([[1, 2], [4, 8]], np.float32))
    b = bf(np.array([[0, 0.5], [0.25, 0]], np.float32))
    got = O.dequant(codes, s, b)
    want = np.array([[1.0] * 64 + [2.5] * 64, [4.25] * 64 + [8.0] * 64])
    assert got.shape == want.shape and np.array_equal(got, want)


def check_dequant8_golden():
    """8-bit variant: hand-worked words, four codes each, lowest byte first."""
    n = 0
    for ln in _lines("dequant8_cases.txt"):
        tok = ln.split()
        word = np.array([[int(tok[0], 16)] * 16], dtype=np.uint32)     # one row, 64 columns
        s = bf(np.array([[float(tok[1])]], np.float32))
        b = bf(np.array([[float(tok[2])]], np.float32))
        want = np.array([float(v) for v in tok[3:7]])
        got = O.dequant(word, s, b, bits=8)
        assert got.shape == (1, 64)
        assert np.array_equal(got[0, :4], want), (tok[0], got[0, :4], want)
        assert np.array_equal(got[0, 60:64], want)
        n += 1
    assert n == 6


def check_dequant8_group_axis():
    """8-bit: 2 rows x 128 columns (32 words per row, two groups per row),
    every code 3: w = 3 s + b of the group (row r, column c // 64)."""
    codes = np.full((2, 32), 0x03030303, dtype=np.uint32)
    s = bf(np.array([[1, 2], [4, 8]], np.float32))
    b = bf(np.array([[0, 0.5], [0.25, 0]], np.float32))
    got = O.dequant(codes, s, b, bits=8)
    want = np.array([[3.0] * 64 + [6.5] * 64, [12.25] * 64 + [24.0] * 64])
    assert got.shape == want.shape and np.array_equal(got, want)


def check_formats_agree():
    """The same codes 0..15 packed eight per word (4 bits) and four per word
    (8 bits) reconstruct the same matrix: the two unpackings agree on which
    column each code belongs to."""
    rng = np.random.default_rng(7)
    q = rng.integers(0, 16, size=(3, 128)).astype(np.uint32)
    w4 = np.zeros((3, 16), np.uint32)
    for i in range(8):
        w4 |= q[:, i::8] << np.uint32(4 * i)
    w8 = np.zeros((3, 32), np.uint32)
    for i in range(4):
        w8 |= q[:, i::4] << np.uint32(8 * i)
    s = bf(rng.uniform(0.01, 0.1, size=(3, 2)).astype(np.float32))
    b = bf(rng.uniform(-1, 1, size=(3, 2)).astype(np.float32))
    a4, a8 = O.dequant(w4, s, b), O.dequant(w8, s, b, bits=8)
    assert np.array_equal(a4, a8)
    assert np.array_equal(O.unpack_codes(w8, 8), q.astype(np.uint8))


def check_e4m3_golden():
    """FP8 E4M3 code values worked by hand from the format's fields."""
    n = 0
    for ln in _lines("e4m3_cases.txt"):
        code, val = ln.split()
        got = O.e4m3_value(np.array([int(code, 16)], np.uint8))[0]
        if val == "nan":
            assert np.isnan(got), code
        else:
            want = float(val)
            assert got == want and np.signbit(got) == np.signbit(want), (code, got, want)
        n += 1
    assert n == 21


def check_e4m3_library():
    """All 256 E4M3 codes against an independent implementation of the same
    format: PyTorch's float8_e4m3fn type (bytes viewed as that type, widened)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    codes = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_value(codes)
    assert np.array_equal(np.isnan(got), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(got[ok], lib[ok]) and np.array_equal(np.signbit(got[ok]), np.signbit(lib[ok]))


def check_e4m3_monotone():
    """Invariant of the format: codes 0x00..0x7E are the non-negative finite
    values in strictly increasing order, and the sign bit only negates."""
    v = O.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0) and v[0] == 0.0 and v[-1] == 448.0
    neg = O.e4m3_value(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -v)


def check_dequant_e4m3_golden():
    """w = s*v(q) + b for hand-worked words of four E4M3 codes, lowest byte first."""
    n = 0
    for ln in _lines("dequant_e4m3_cases.txt"):
        tok = ln.split()
        word = np.array([[int(tok[0], 16)] * 16], dtype=np.uint32)     # one row, 64 columns
        s = bf(np.array([[float(tok[1])]], np.float32))
        b = bf(np.array([[float(tok[2])]], np.float32))
        want = np.array([float(v) for v in tok[3:7]])
        got = O.dequant(word, s, b, bits=8, fmt=O.CODES_E4M3)
        assert got.shape == (1, 64)
        assert np.array_equal(got[0, :4], want), (tok[0], got[0, :4], want)
        assert np.array_equal(got[0, 60:64], want)
        n += 1
    assert n == 4


def check_e4m3_layer_integers():
    """A layer whose codes are the E4M3 encodings of integers 0..15 (encoded by
    PyTorch's float8_e4m3fn, exact for these integers) computes the same output
    as the unsigned 8-bit layer with those integers as codes: the format only
    changes how a code is read."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    L, x = S.draw_config("w8_tiny_T4")
    lut = torch.arange(256, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy().astype(np.uint32)

    def small_ints(m):
        q = O.unpack_codes(m.codes, 8) & 15                         # integer codes 0..15
        w_int = np.zeros(m.codes.shape, np.uint32)
        w_fp8 = np.zeros(m.codes.shape, np.uint32)
        for i in range(4):
            w_int |= q[..., i::4].astype(np.uint32) << np.uint32(8 * i)
            w_fp8 |= lut[q[..., i::4]] << np.uint32(8 * i)
        return S.W4Matrix(w_int, m.scales, m.biases), S.W4Matrix(w_fp8, m.scales, m.biases)

    names = ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")
    pairs = {n: small_ints(getattr(L, n)) for n in names}
    import dataclasses
    Li = dataclasses.replace(L, **{n: pairs[n][0] for n in names})
    Lf = dataclasses.replace(L, code_format=S.CODES_E4M3, **{n: pairs[n][1] for n in names})
    ri, rf = O.moe_layer(Li, x), O.moe_layer(Lf, x)
    assert np.array_equal(ri["out"], rf["out"])
    # and the format is really read: the same words read as unsigned bytes differ
    Lu = dataclasses.replace(Lf, code_format=S.CODES_UINT)
    assert not np.allclose(O.moe_layer(Lu, x)["out"], rf["out"])


def check_format_size():
    """Section "Dequantise weights during matrix multiplication": a 35B-parameter
    model shrinks from about 70 GB of bf16 to a 19.4 GB checkpoint.  One bf16
    scale and one bf16 bias per 64 weights cost 0.5 bit per weight on top of the
    4-bit code: 4.5 bits -> 19.7 GB, within 2% of the quoted size (the
    checkpoint also keeps some tensors unquantised and counts in GB vs GiB)."""
    bpw = O.bits_per_weight()
    assert bpw == 4.5
    gb = O.checkpoint_gb(35e9, bpw)
    assert abs(gb - 19.4) / 19.4 < 0.02, gb
    assert abs(O.checkpoint_gb(35e9, 16) - 70.0) < 1e-9
    # of the usual group sizes, 64 is the one that lands nearest the quoted size
    err = {g: abs(O.checkpoint_gb(35e9, O.bits_per_weight(g)) - 19.4) for g in (16, 32, 64, 128, 256)}
    assert min(err, key=err.get) == 64, err


# ---------------------------------------------------------------------------
# router
# ---------------------------------------------------------------------------
def _router_fixture():
    W, G, cases = [], None, []
    for ln in _lines("router_tiny.txt"):
        tok = ln.split()
        if tok[0] in ("W0", "W1"):
            W.append([float(v) for v in tok[1:]])
        elif tok[0] == "G":
            G = np.array([float(v) for v in tok[1:]])
        else:
            head, idx, w, gam = [p.split() for p in ln.split("|")]
            x = np.array([float(head[1]), float(head[2])])
            if head[3] == "-":
                bias, k = None, int(head[4])
            else:
                bias, k = np.array([float(v) for v in head[3:7]]), int(head[7])
            cases.append((head[0], x, bias, k, [int(v) for v in idx], [float(v) for v in w], float(gam[0])))
    return np.array(W), G, cases


def check_router_golden():
    W, G, cases = _router_fixture()
    assert len(cases) == 5
    for name, x, bias, k, idx, w, gam in cases:
        ri, rw, rg, _ = O.route(x[None, :], W, bias, G, k)
        assert list(ri[0]) == idx, (name, ri[0], idx)
        assert np.allclose(rw[0], w, rtol=0, atol=1e-15), (name, rw[0], w)
        assert abs(rg[0] - gam) < 1e-15, (name, rg[0], gam)


def check_router_invariants(seed=0):
    rng = np.random.default_rng(seed)
    H, E = 32, 16
    x = rng.normal(size=(40, H))
    W = rng.normal(0, 0.3, size=(H, E))
    g = rng.normal(0, 0.3, size=H)
    for k in (1, 3, 8, E):
        idx, w, gam, l = O.route(x, W, None, g, k)
        assert np.allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
        # selection = the k largest scores, by descending score (library sort)
        ref = np.argsort(-l, axis=1, kind="stable")[:, :k]
        assert np.array_equal(idx, ref)
        if k == 1:
            assert np.all(w == 1.0)
        if k == E:
            # k = E reduces to dense softmax gating
            dense = scipy.special.softmax(l, axis=1)
            assert np.allclose(np.take_along_axis(dense, idx, 1), w, rtol=0, atol=1e-14)
        # equals softmax over all experts renormalised over the selection
        full = scipy.special.softmax(l, axis=1)
        sel = np.take_along_axis(full, idx, 1)
        assert np.allclose(sel / sel.sum(1, keepdims=True), w, rtol=0, atol=1e-14)
    assert np.allclose(gam, scipy.special.expit(x @ g), rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# grouping
# ---------------------------------------------------------------------------
def check_group_golden():
    n = 0
    for ln in _lines("group_tiny.txt"):
        parts = [p.strip() for p in ln.split("|")]
        E, k = [int(v) for v in parts[1].split()]
        idx = np.array([[int(v) for v in r.split()] for r in parts[2].split(";")])
        assert idx.shape[1] == k
        want = [np.array([int(v) for v in p.split()]) for p in parts[3:7]]
        got = O.group(idx, E)
        for g, w_, nm in zip(got, want, ("counts", "offsets", "perm", "inv")):
            assert np.array_equal(g, w_), (parts[0], nm, g, w_)
        n += 1
    assert n == 3


def check_block_map_golden():
    """The block list by its exact (expert, first row) entries, hand-worked."""
    n = 0
    for ln in _lines("block_map_tiny.txt"):
        parts = [p.strip() for p in ln.split("|")]
        B = int(parts[1])
        counts = np.array([int(v) for v in parts[2].split()])
        want = [] if parts[3] == "-" else [tuple(int(v) for v in b.split()) for b in parts[3].split(";")]
        got = [(int(e), int(r)) for e, r in O.block_map(counts, B)]
        assert got == want, (parts[0], got, want)
        n += 1
    assert n == 5


def check_group_invariants(seed=1):
    rng = np.random.default_rng(seed)
    for T, E, k in ((1, 4, 2), (37, 16, 4), (200, 64, 8)):
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        counts, offsets, perm, inv = O.group(idx, E)
        assert counts.sum() == T * k and offsets[-1] == T * k and offsets[0] == 0
        assert np.array_equal(np.sort(perm), np.arange(T * k))           # bijection
        assert np.array_equal(inv[perm], np.arange(T * k))               # inv o perm = id
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(idx.reshape(-1)[seg] == e)
            assert np.all(np.diff(seg // k) > 0)                         # ascending tokens
        bc, bo, bp, bi = BF.grouping(idx.tolist(), E)                    # brute force
        assert list(counts) == bc and list(offsets) == bo and list(perm) == bp and list(inv) == bi
        blocks = O.block_map(counts, 16)
        assert len(blocks) == sum(-(-int(c) // 16) for c in counts)


# ---------------------------------------------------------------------------
# expert FFN and whole layer
# ---------------------------------------------------------------------------
def check_silu():
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(O.silu(-2.0) - (-2.0 / (1.0 + math.exp(2.0)))) < 1e-16
    assert abs(O.silu(40.0) - 40.0) < 1e-12 and abs(O.silu(-40.0)) < 1e-12


def _w4_from_codes(q, s=1.0, b=0.0):
    """Pack an integer code matrix q [rows][cols] (0..15) with one scale/bias."""
    rows, cols = q.shape
    words = np.zeros((rows, cols // 8), dtype=np.uint32)
    for i in range(8):
        words |= (q[:, i::8].astype(np.uint32) << np.uint32(4 * i))
    sc = bf(np.full((rows, cols // 64), s, np.float32))
    bi = bf(np.full((rows, cols // 64), b, np.float32))
    return S.W4Matrix(words, sc, bi)


def check_structured_ffn():
    """Shift matrices make every output a closed form: with Wg[i, (i+1)%n] = 1,
    Wu = identity and Wd[o, (o+2)%n] = 1 the FFN gives
    y[o] = silu(x[(o+3)%n]) * x[(o+2)%n]."""
    n = 64
    ar = np.arange(n)
    qg = np.zeros((n, n), np.int64); qg[ar, (ar + 1) % n] = 1
    qu = np.eye(n, dtype=np.int64)
    qd = np.zeros((n, n), np.int64); qd[ar, (ar + 2) % n] = 1
    mg, mu, md = _w4_from_codes(qg), _w4_from_codes(qu), _w4_from_codes(qd)
    x = (ar / 8.0 - 3.0)[None, :]
    y = O.expert_ffn(x, O.dequant(mg.codes, mg.scales, mg.biases), O.dequant(mu.codes, mu.scales, mu.biases),
                     O.dequant(md.codes, md.scales, md.biases))
    for o in range(n):
        a, c = x[0, (o + 3) % n], x[0, (o + 2) % n]
        assert abs(y[0, o] - a / (1.0 + math.exp(-a)) * c) < 1e-13, o


def _const_layer():
    """The closed-form layer of layer_tiny.txt (H = I = 64, E = 2, k = 1, s = 0)."""
    H = I = 64

    def mat(rows, cols, bval, lead=()):
        codes = np.full(lead + (rows, cols // 8), 0x76543210, dtype=np.uint32)   # codes irrelevant: s = 0
        sc = bf(np.zeros(lead + (rows, cols // 64), np.float32))
        bi = bf(np.full(lead + (rows, cols // 64), bval, np.float32))
        return S.W4Matrix(codes, sc, bi)

    def stack(a, b):
        return S.W4Matrix(np.stack([a.codes, b.codes]), np.stack([a.scales, b.scales]), np.stack([a.biases, b.biases]))

    p6, p5 = 2.0 ** -6, 2.0 ** -5
    gate = stack(mat(I, H, p6), mat(I, H, -p6))
    up = stack(mat(I, H, p5), mat(I, H, -p5))
    down = stack(mat(H, I, p6), mat(H, I, -p6))
    rw = np.zeros((H, 2), np.float32); rw[:, 0] = p6
    return S.W4Layer(H, 2, I, 1, rw, None, np.full(H, p6, np.float32), gate, up, down,
                     mat(I, H, p5), mat(I, H, -p6), mat(H, I, p5))


def check_layer_golden():
    L = _const_layer()
    rows = list(_lines("layer_tiny.txt"))
    assert len(rows) == 2
    x = bf(np.stack([np.ones(64, np.float32), -np.ones(64, np.float32)]))
    r = O.moe_layer(L, x)
    for ln in rows:
        t, e, val, bits = ln.split()
        t = int(t)
        assert r["idx"][t, 0] == int(e)
        assert np.allclose(r["out"][t], float(val), rtol=0, atol=1e-14), (t, r["out"][t, :2], val)
        assert np.all(r["out_bf16"][t] == int(bits, 16))


def check_identical_experts(seed=2):
    """All routed experts equal => the output no longer depends on the routing,
    because the weights sum to one: out = y(x) + gamma * y_shared."""
    L, x = S.draw_config("tiny_T4")
    for m in (L.gate, L.up, L.down):
        for a in (m.codes, m.scales, m.biases):
            a[:] = a[0:1]
    r = O.moe_layer(L, x)
    xf = O.bf16_to_f64(x)
    y = O.expert_ffn(xf, *[O.dequant(m.codes[0], m.scales[0], m.biases[0]) for m in (L.gate, L.up, L.down)])
    ysh = O.expert_ffn(xf, *[O.dequant(m.codes, m.scales, m.biases) for m in (L.sh_gate, L.sh_up, L.sh_down)])
    gam = scipy.special.expit(xf @ L.shared_gate.astype(np.float64))
    assert np.allclose(r["out"], y + gam[:, None] * ysh, rtol=1e-12, atol=1e-12)


def check_dense_gating():
    """k = E: out = sum_e softmax(l)_e y_e(x) + gamma y_shared (library softmax)."""
    L, x = S.draw_config("tiny_T4")
    L.top_k = L.E
    r = O.moe_layer(L, x)
    xf = O.bf16_to_f64(x)
    l = xf @ L.router_w.astype(np.float64)
    p = scipy.special.softmax(l, axis=1)
    out = np.zeros_like(xf)
    for e in range(L.E):
        out += p[:, e:e + 1] * O.expert_ffn(xf, *[O.dequant(m.codes[e], m.scales[e], m.biases[e])
                                                  for m in (L.gate, L.up, L.down)])
    ysh = O.expert_ffn(xf, *[O.dequant(m.codes, m.scales, m.biases) for m in (L.sh_gate, L.sh_up, L.sh_down)])
    out += scipy.special.expit(xf @ L.shared_gate.astype(np.float64))[:, None] * ysh
    assert np.allclose(r["out"], out, rtol=1e-12, atol=1e-12)


def check_brute_force_tiny():
    L, x = S.draw_config("tiny_T4")
    r = O.moe_layer(L, x)
    outs, sel = BF.layer(L, x)
    ref = np.array(outs)
    assert np.max(np.abs(r["out"] - ref)) <= 1e-12 * np.max(np.abs(ref))
    for t, (order, w, gam) in enumerate(sel):
        assert list(r["idx"][t]) == order
        assert np.allclose(r["w"][t], w, rtol=0, atol=1e-14) and abs(r["gamma"][t] - gam) < 1e-14


def check_row_independence():
    L, x = S.draw_config("tiny_T4", T=12)
    full = O.moe_layer(L, x)
    for a, b in ((0, 4), (4, 8), (8, 12)):
        part = O.moe_layer(L, x[a:b])
        assert np.allclose(part["out"], full["out"][a:b], rtol=1e-14, atol=1e-14)
        assert np.array_equal(part["idx"], full["idx"][a:b])


PINS = [check_dequant_golden, check_group_axis, check_dequant8_golden, check_dequant8_group_axis,
        check_formats_agree, check_e4m3_golden, check_e4m3_library, check_e4m3_monotone,
        check_dequant_e4m3_golden, check_e4m3_layer_integers, check_format_size, check_router_golden,
        check_router_invariants, check_group_golden, check_block_map_golden, check_group_invariants, check_silu,
        check_structured_ffn, check_layer_golden, check_identical_experts, check_dense_gating,
        check_brute_force_tiny, check_row_independence]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


def test_generator_distribution():
    """The generator draws the distributions it states (codes uniform 0..15,
    s = |N(0, 0.02)|, b = -8 s + N(0, 0.002)) and honours the score margin."""
    L, x = S.draw_config("tiny_T4", T=64)
    q = O.unpack_codes(L.gate.codes).ravel()
    cnt = np.bincount(q, minlength=16)
    assert cnt.min() > 0.8 * q.size / 16 and cnt.max() < 1.2 * q.size / 16
    s = O.bf16_to_f64(L.gate.scales).ravel()
    b = O.bf16_to_f64(L.gate.biases).ravel()
    assert np.all(s >= 0) and abs(s.mean() - 0.02 * math.sqrt(2 / math.pi)) < 2e-3
    assert abs(np.std(b + 8 * s) - 0.002) < 5e-4
    l = O.router_scores(O.bf16_to_f64(x), L.router_w, L.router_bias)
    lead = -np.sort(-l, axis=1)[:, :L.top_k + 1]
    assert np.all(lead[:, :-1] - lead[:, 1:] >= S.MARGIN)
    # the 8-bit variant: codes uniform 0..255, s = |N(0, 0.02)| / 17, b = -128 s + N(0, 0.002)
    L8, _ = S.draw_config("w8_tiny_T4")
    assert L8.code_bits == 8 and L8.gate.codes.shape[-1] == L8.H // 4
    q8 = O.unpack_codes(L8.gate.codes, 8).ravel()
    cnt8 = np.bincount(q8, minlength=256)
    assert cnt8.min() > 0.6 * q8.size / 256 and cnt8.max() < 1.4 * q8.size / 256
    s8 = O.bf16_to_f64(L8.gate.scales).ravel()
    b8 = O.bf16_to_f64(L8.gate.biases).ravel()
    assert np.all(s8 >= 0) and abs(s8.mean() - 0.02 / 17 * math.sqrt(2 / math.pi)) < 2e-4
    assert abs(np.std(b8 + 128 * s8) - 0.002) < 5e-4
    # FP8 E4M3 codes: uniform sign, exponent field 3..10, uniform mantissa; never NaN;
    # s = |N(0, 0.02)|, b = N(0, 0.002)
    Lf, _ = S.draw_config("e4m3_tiny_T4")
    assert Lf.code_bits == 8 and Lf.code_format == S.CODES_E4M3
    qf = O.unpack_codes(Lf.gate.codes, 8).ravel().astype(np.int64)
    ef = (qf >> 3) & 15
    assert ef.min() == 3 and ef.max() == 10
    assert abs(np.mean(qf >> 7) - 0.5) < 0.05
    assert np.bincount(qf & 7, minlength=8).min() > 0.8 * qf.size / 8
    assert not np.any(np.isnan(O.e4m3_value(qf.astype(np.uint8))))
    sf = O.bf16_to_f64(Lf.gate.scales).ravel()
    bfv = O.bf16_to_f64(Lf.gate.biases).ravel()
    assert np.all(sf >= 0) and abs(sf.mean() - 0.02 * math.sqrt(2 / math.pi)) < 2e-3
    assert abs(np.std(bfv) - 0.002) < 5e-4


# ---------------------------------------------------------------------------
# planted mistakes: each broken oracle must fail at least one pin
# ---------------------------------------------------------------------------
def _reversed_nibbles(words, bits=4):
    if bits != 4:
        return _UNPACK(words, bits)
    w = np.asarray(words, dtype=np.uint32)
    nib = np.stack([(w >> np.uint32(4 * (7 - i))) & np.uint32(0xF) for i in range(8)], axis=-1)
    return nib.reshape(w.shape[:-1] + (w.shape[-1] * 8,)).astype(np.uint8)


def _reversed_bytes(words, bits=4):
    if bits != 8:
        return _UNPACK(words, bits)
    w = np.asarray(words, dtype=np.uint32)
    c = np.stack([(w >> np.uint32(8 * (3 - i))) & np.uint32(0xFF) for i in range(4)], axis=-1)
    return c.reshape(w.shape[:-1] + (w.shape[-1] * 4,)).astype(np.uint8)


def _swapped_affine(codes, scales, biases, bits=4, fmt=0):
    q = O.unpack_codes(codes, bits).astype(np.float64)
    s = np.repeat(O.bf16_to_f64(scales), 64, axis=-1)
    b = np.repeat(O.bf16_to_f64(biases), 64, axis=-1)
    return b * q + s


def _groups_down_rows(codes, scales, biases, bits=4, fmt=0):
    q = O.unpack_codes(codes, bits).astype(np.float64)
    s = np.repeat(np.swapaxes(O.bf16_to_f64(scales), -1, -2), 64, axis=-1)   # group index on the wrong axis
    b = np.repeat(np.swapaxes(O.bf16_to_f64(biases), -1, -2), 64, axis=-1)
    return s * q + b


_E4M3 = O.e4m3_value


def _e4m3_bias_8(q):
    """E4M3 read with exponent bias 8 (the E5M2-style bias mistake)."""
    return _E4M3(q) / 2.0


def _e4m3_no_subnormals(q):
    """E4M3 with the implicit leading one also at exponent field 0."""
    v = _E4M3(q)
    qq = np.asarray(q, np.uint8).astype(np.int64)
    sub = ((qq >> 3) & 0xF) == 0
    return np.where(sub, np.where(qq & 0x80, -1.0, 1.0) * (1.0 + (qq & 7) / 8.0) * 2.0 ** -7, v)


def _e4m3_unsigned(q):
    """E4M3 with the sign bit ignored."""
    return np.abs(_E4M3(q))


def _unrenormalised_route(x, W, bias, g, k):
    l = O.router_scores(x, W, bias)
    idx = np.stack([O.select_top_k(r, k) for r in l])
    full = scipy.special.softmax(l, axis=1)
    return idx, np.take_along_axis(full, idx, 1), O.sigmoid(np.asarray(x) @ np.asarray(g)), l


def _ties_to_higher(row, k):
    order = sorted(range(len(row)), key=lambda e: (-row[e], -e))
    return order[:k]


def _silu_on_up(xr, wg, wu, wd):
    return (O.silu(xr @ wu.T) * (xr @ wg.T)) @ wd.T


def _down_transposed(xr, wg, wu, wd):
    return (O.silu(xr @ wg.T) * (xr @ wu.T)) @ wd


def _group_by_slot(idx, E):
    T, k = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    fill = offsets[:-1].copy()
    perm = np.zeros(T * k, np.int64); inv = np.zeros(T * k, np.int64)
    for j in range(k):                  # slot-major instead of token-major
        for t in range(T):
            e = idx[t, j]; p = fill[e]; fill[e] += 1
            perm[p] = t * k + j; inv[t * k + j] = p
    return counts, offsets, perm, inv


def _ungated_sigmoid(z):
    return np.ones_like(np.asarray(z, dtype=np.float64)) if np.ndim(z) else 1.0


def _block_map_short_stride(counts, rows_per_block):
    blocks = []
    for e, c in enumerate(counts):
        for r0 in range(0, int(c), max(1, rows_per_block - 1)):
            blocks.append((e, r0))
    return blocks


def _block_map_row_major(counts, rows_per_block):
    blocks = []
    for r0 in range(0, int(max(counts, default=0)), rows_per_block):
        for e, c in enumerate(counts):
            if r0 < c:
                blocks.append((e, r0))
    return blocks


_UNPACK = O.unpack_codes

MUTANTS = [
    ("unpack_codes", _reversed_nibbles),
    ("unpack_codes", _reversed_bytes),
    ("e4m3_value", _e4m3_bias_8),
    ("e4m3_value", _e4m3_no_subnormals),
    ("e4m3_value", _e4m3_unsigned),
    ("dequant", _swapped_affine),
    ("dequant", _groups_down_rows),
    ("route", _unrenormalised_route),
    ("select_top_k", _ties_to_higher),
    ("expert_ffn", _silu_on_up),
    ("expert_ffn", _down_transposed),
    ("group", _group_by_slot),
    ("block_map", _block_map_short_stride),
    ("block_map", _block_map_row_major),
    ("sigmoid", _ungated_sigmoid),
]


@pytest.mark.parametrize("name,fn", MUTANTS, ids=[f"{n}:{f.__name__}" for n, f in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)
    failed = []
    for pin in PINS:
        if pin in (check_brute_force_tiny,):
            continue                      # slowest pin; the others must already catch it
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name}:{fn.__name__}"


def test_tolerance_reading():
    """The bf16 output format alone breaks the literal max bound on this
    workload: the exact result rounded to bf16 is off by up to 2^-8 of a value
    that reaches ~9 rms.  The adopted reading (error beyond half a bf16 ulp)
    gives that rounding exactly zero excess, and the L2 bound holds as stated."""
    from tests import tolerance as TOL
    L, x = S.draw_config("prefill_T512", T=128)
    ref = O.moe_layer(L, x)["out"]
    rounded = O.bf16_to_f64(O.f64_to_bf16(ref))
    m = TOL.metrics(rounded, ref)
    assert m["max_rel_literal"] > TOL.MAX_REL          # literal bar unattainable for bf16 output
    assert m["max_rel"] <= 0.0 and m["l2"] < 2e-3      # reading: final rounding costs nothing
    # half-ulp bound of a bf16 rounding (the oracle rounds via fp32: the double
    # rounding may add at most one fp32 half-ulp, 2^-16 of a bf16 half-ulp)
    v = np.random.default_rng(0).normal(size=100000) * np.exp(np.random.default_rng(1).normal(size=100000) * 3)
    assert np.all(np.abs(O.bf16_to_f64(O.f64_to_bf16(v)) - v) <= TOL.halfulp_bf16(v) * (1 + 2.0 ** -15))
