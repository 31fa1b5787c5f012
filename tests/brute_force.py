"""Pure-Python brute force of the layer for tiny shapes (a pin for the oracle).

Written with scalar loops and the math module only: bit extraction per code,
score sums, selection by sorting (score, index) pairs, softmax with math.exp,
grouping by scanning every (expert, token) pair, and the SwiGLU FFN as nested
sums.  It shares no code with the oracle; it follows the same pages:
"Optimizing on-device inference for Apple Silicon", sections "Qwen creates
three different workload shapes", "Dequantise weights during matrix
multiplication", "Keep expert routing on the GPU", "Reduce intermediate state
and traffic".
"""
import math
import struct


def bf16(bits):
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def weight(codes, scales, biases, r, c):
    word = int(codes[r][c // 8])
    q = (word >> (4 * (c % 8))) & 15
    return bf16(scales[r][c // 64]) * q + bf16(biases[r][c // 64])


def ffn(x, gm, um, dm, H, I):
    h = []
    for i in range(I):
        g = sum(x[c] * weight(gm.codes, gm.scales, gm.biases, i, c) for c in range(H))
        u = sum(x[c] * weight(um.codes, um.scales, um.biases, i, c) for c in range(H))
        h.append(g / (1.0 + math.exp(-g)) * u)
    return [sum(h[i] * weight(dm.codes, dm.scales, dm.biases, o, i) for i in range(I)) for o in range(H)]


class _Sub:
    def __init__(self, m, e):
        self.codes, self.scales, self.biases = m.codes[e], m.scales[e], m.biases[e]


def layer(L, x_bits):
    H, E, I, k = L.H, L.E, L.I, L.top_k
    outs, sel_all = [], []
    for xt in x_bits:
        x = [bf16(v) for v in xt]
        sc = []
        for e in range(E):
            s = sum(x[h] * float(L.router_w[h][e]) for h in range(H))
            if L.router_bias is not None:
                s += float(L.router_bias[e])
            sc.append(s)
        order = sorted(range(E), key=lambda e: (-sc[e], e))[:k]
        m = max(sc[e] for e in order)
        z = sum(math.exp(sc[e] - m) for e in order)
        w = [math.exp(sc[e] - m) / z for e in order]
        gam = 1.0 / (1.0 + math.exp(-sum(x[h] * float(L.shared_gate[h]) for h in range(H))))
        out = [0.0] * H
        for e, we in zip(order, w):
            y = ffn(x, _Sub(L.gate, e), _Sub(L.up, e), _Sub(L.down, e), H, I)
            out = [a + we * b for a, b in zip(out, y)]
        ysh = ffn(x, L.sh_gate, L.sh_up, L.sh_down, H, I)
        outs.append([a + gam * b for a, b in zip(out, ysh)])
        sel_all.append((order, w, gam))
    return outs, sel_all


def grouping(idx, E):
    T, k = len(idx), len(idx[0])
    counts = [sum(1 for t in range(T) for j in range(k) if idx[t][j] == e) for e in range(E)]
    offsets = [sum(counts[:e]) for e in range(E + 1)]
    perm = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t][j] == e:
                    perm.append(t * k + j)
    inv = [0] * (T * k)
    for p, a in enumerate(perm):
        inv[a] = p
    return counts, offsets, perm, inv
