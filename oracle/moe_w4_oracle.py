"""CPU oracle for the W4 group-affine sparse-MoE layer.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
the CPU-baseline leg of the benchmark may import this module.  The CUDA
library never calls it, and it shares no code, header, table or helper with
the CUDA path.

The layer follows "Optimizing on-device inference for Apple Silicon"
(perplexity.ai blog, Chinese edition):
  * section "Qwen creates three different workload shapes": the router scores
    256 experts per token and keeps 8; one shared expert processes every token;
  * section "Dequantise weights during matrix multiplication": each weight is a
    4-bit integer code, and each group of 64 weights shares one bf16 scale and
    one bf16 bias that reconstruct its value; accumulation is 32-bit float and
    the output is bf16;
  * section "Keep expert routing on the GPU": histogram of assignments per
    expert -> prefix scan to start offsets -> scatter of rows into expert
    groups -> list of fixed-size blocks;
  * section "Reduce intermediate state and traffic": the expert output
    projection is combined with the routing scores and the shared expert's
    result.
The pages leave the arithmetic details open; this oracle takes these readings
(each one also stated where it is used):
  R1  w = s*q + b with q the unsigned code 0..15;
  R2  eight codes per uint32, lowest input column in the lowest nibble;
  R3  a group is 64 consecutive input columns of one output row;
  R4  routing weights are the softmax over the k selected scores (equal to a
      softmax over all experts renormalised over the selection);
  R5  equal scores select the lower expert index first; the selection is
      listed by descending score;
  R6  the shared expert is scaled by gamma = sigmoid(x . g);
  R7  expert FFN is SwiGLU: h = silu(x Wg^T) * (x Wu^T), y = h Wd^T,
      silu(z) = z * sigmoid(z);
  R8  rows of one expert group are ordered by ascending token index;
  R9  out = sum_j w_j y_{e_j} + gamma * y_shared, rounded once to bf16;
  R10 the 8-bit affine variant (a weight-format variant of the same layer: MLX
      affine quantisation with group size 64, with which an encoder's linear
      layers are quantised at 8 and 4 bits in "Engineering investigation: can
      this MLX port be 10x faster?", section "Selective quantisation") keeps
      R1 and R3 with q the unsigned code 0..255, four codes per uint32,
      lowest input column in the lowest byte;
  R11 the FP8 E4M3 variant (the news item on the lithos-metal pull requests
      names an "FP8 E4M3 decode" that handles two codes per half2; it gives
      nothing else) stores each weight's code as one FP8 E4M3 byte, laid out
      as in R10, and keeps the group scale and bias: w = s*v(q) + b with v(q)
      the value of the byte in the E4M3 format of "FP8 Formats for Deep
      Learning" (Micikevicius et al., 2022): sign bit, 4 exponent bits with
      bias 7, 3 mantissa bits, subnormals at exponent field 0, no infinities,
      and NaN only at exponent and mantissa fields all ones.

Everything is float64; the only rounding to bf16 is the final output (and it
goes float64 -> float32 -> bf16, a double rounding that is far below any
tolerance used against it).  Parity pins: see tests/test_oracle_pins.py.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

GROUP = 64


# ----------------------------------------------------------------------------
# number formats
# ----------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """float64 -> bfloat16 bits, via float32, round to nearest even."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------
# group-affine 4-bit weights (section "Dequantise weights during matrix
# multiplication"; readings R1-R3)
# ----------------------------------------------------------------------------
def unpack_codes(words: np.ndarray, bits: int = 4) -> np.ndarray:
    """uint32 [..., n] -> uint8 codes [..., (32/bits) n].  4 bits: column 8*w + i
    is nibble i of word w, nibble 0 being the lowest four bits (R2); 8 bits:
    column 4*w + i is byte i of word w, byte 0 the lowest (R10)."""
    assert bits in (4, 8)
    per = 32 // bits
    mask = np.uint32((1 << bits) - 1)
    w = np.asarray(words, dtype=np.uint32)
    c = np.stack([(w >> np.uint32(bits * i)) & mask for i in range(per)], axis=-1)
    return c.reshape(w.shape[:-1] + (w.shape[-1] * per,)).astype(np.uint8)


CODES_UINT = 0      # layer code_format: unsigned integer codes
CODES_E4M3 = 1      # layer code_format: FP8 E4M3 codes (R11)


def e4m3_value(q) -> np.ndarray:
    """FP8 E4M3 bytes -> float64 (R11).  Fields: sign S = bit 7, exponent
    field e = bits 6..3, mantissa field m = bits 2..0.  e = 0: (-1)^S m/8 2^-6
    (subnormal; m = 0 is a signed zero); otherwise (-1)^S (1 + m/8) 2^(e-7);
    e = 15 with m = 7 is NaN.  The largest finite magnitude is 1.75 * 2^8 = 448."""
    q = np.asarray(q, dtype=np.uint8).astype(np.int64)
    sign = np.where(q & 0x80, -1.0, 1.0)
    e = (q >> 3) & 0xF
    m = (q & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    return np.where((e == 15) & (q & 0x7 == 7), np.nan, sign * mag)


def dequant(codes: np.ndarray, scales: np.ndarray, biases: np.ndarray, bits: int = 4,
            fmt: int = CODES_UINT) -> np.ndarray:
    """Reconstruct a [rows][cols] matrix in float64: w[r, c] = s[r, c//64] * q[r, c]
    + b[r, c//64] (R1, R3; R10 for 8-bit codes), with q replaced by the E4M3
    value of the code for FP8 codes (R11)."""
    if fmt == CODES_E4M3:
        assert bits == 8
        q = e4m3_value(unpack_codes(codes, 8))
    else:
        q = unpack_codes(codes, bits).astype(np.float64)
    s = np.repeat(bf16_to_f64(scales), GROUP, axis=-1)
    b = np.repeat(bf16_to_f64(biases), GROUP, axis=-1)
    assert q.shape == s.shape == b.shape, (q.shape, s.shape)
    return s * q + b


# ----------------------------------------------------------------------------
# router (section "Qwen creates three different workload shapes"; R4-R6)
# ----------------------------------------------------------------------------
def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, dtype=np.float64)))


def router_scores(x: np.ndarray, router_w: np.ndarray, router_bias: Optional[np.ndarray]) -> np.ndarray:
    """Scores l[t, e] = sum_h x[t, h] W_r[h, e] (+ bias[e]), float64."""
    l = np.asarray(x, np.float64) @ np.asarray(router_w, np.float64)
    if router_bias is not None:
        l = l + np.asarray(router_bias, np.float64)[None, :]
    return l


def select_top_k(scores_row: np.ndarray, k: int) -> list:
    """Indices of the k largest scores, largest first; on equal scores the lower
    index comes first (R5).  Repeated selection of the best remaining expert."""
    remaining = list(range(len(scores_row)))
    chosen = []
    for _ in range(k):
        best = remaining[0]
        for e in remaining[1:]:
            if scores_row[e] > scores_row[best]:
                best = e
        chosen.append(best)
        remaining.remove(best)
    return chosen


def route(x: np.ndarray, router_w, router_bias, shared_gate, k: int):
    """Per token: selected experts, renormalised softmax weights, shared gate.

    Returns (idx int64 [T][k], w float64 [T][k], gamma float64 [T], scores [T][E]).
    """
    l = router_scores(x, router_w, router_bias)
    T = l.shape[0]
    idx = np.zeros((T, k), dtype=np.int64)
    w = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        sel = select_top_k(l[t], k)
        idx[t] = sel
        top = l[t, sel]
        ex = np.exp(top - top.max())           # softmax over the selection (R4)
        w[t] = ex / ex.sum()
    gamma = sigmoid(np.asarray(x, np.float64) @ np.asarray(shared_gate, np.float64))  # R6
    return idx, w, gamma, l


# ----------------------------------------------------------------------------
# grouping (section "Keep expert routing on the GPU"; R8)
# ----------------------------------------------------------------------------
def group(idx: np.ndarray, E: int):
    """Histogram -> exclusive prefix scan -> stable scatter.

    counts[e]  = number of (t, j) with idx[t, j] == e
    offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
    position of (t, j) = offsets[e] + number of earlier tokens t' < t that also
    selected e (a token selects an expert at most once)
    perm[p] = t*k + j for the assignment at position p; inv = perm^-1.
    """
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    perm = np.zeros(T * k, dtype=np.int64)
    inv = np.zeros(T * k, dtype=np.int64)
    for t in range(T):             # ascending token order gives the stable order
        for j in range(k):
            e = idx[t, j]
            p = fill[e]
            fill[e] += 1
            perm[p] = t * k + j
            inv[t * k + j] = p
    return counts, offsets, perm, inv


def block_map(counts: np.ndarray, rows_per_block: int):
    """Fixed-size blocks the grouped product must process: (expert, first row)
    for every block of `rows_per_block` rows of every non-empty expert group."""
    blocks = []
    for e, c in enumerate(counts):
        for r0 in range(0, int(c), rows_per_block):
            blocks.append((e, r0))
    return blocks


# ----------------------------------------------------------------------------
# expert FFN (R7) and the whole layer (R9)
# ----------------------------------------------------------------------------
def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z * sigmoid(z)


def expert_ffn(xr: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """xr [n][H] float64, wg/wu [I][H], wd [H][I] -> y [n][H]."""
    h = silu(xr @ wg.T) * (xr @ wu.T)
    return h @ wd.T


def _mat(m, e=None, bits=4, fmt=CODES_UINT):
    if e is None:
        return dequant(m.codes, m.scales, m.biases, bits, fmt)
    return dequant(m.codes[e], m.scales[e], m.biases[e], bits, fmt)


def moe_layer(layer, x_bits: np.ndarray, tokens: Optional[np.ndarray] = None):
    """Whole layer for the rows `tokens` of x (all rows if None).

    `layer` carries H, E, I, top_k, router_w, router_bias, shared_gate, the
    six quantised matrices (attributes codes/scales/biases) gate, up, down,
    sh_gate, sh_up, sh_down and, optionally, code_bits (4 when absent) and
    code_format (CODES_UINT when absent).  Returns a dict with out (float64),
    out_bf16 (bits) and the routing / grouping intermediates of the selected
    rows.
    """
    x_all = bf16_to_f64(x_bits)
    rows = np.arange(x_all.shape[0]) if tokens is None else np.asarray(tokens)
    x = x_all[rows]
    k = layer.top_k
    f = (getattr(layer, "code_bits", 4), getattr(layer, "code_format", CODES_UINT))
    idx, w, gamma, scores = route(x, layer.router_w, layer.router_bias, layer.shared_gate, k)
    out = np.zeros_like(x)
    for e in np.unique(idx):
        sel_t, sel_j = np.nonzero(idx == e)
        y = expert_ffn(x[sel_t], _mat(layer.gate, e, *f), _mat(layer.up, e, *f), _mat(layer.down, e, *f))
        out[sel_t] += w[sel_t, sel_j][:, None] * y
    y_sh = expert_ffn(x, _mat(layer.sh_gate, None, *f), _mat(layer.sh_up, None, *f),
                      _mat(layer.sh_down, None, *f))
    out += gamma[:, None] * y_sh
    res = dict(out=out, out_bf16=f64_to_bf16(out), idx=idx, w=w, gamma=gamma, scores=scores)
    if tokens is None:
        counts, offsets, perm, inv = group(idx, layer.E)
        res.update(counts=counts, offsets=offsets, perm=perm, inv=inv)
    return res


# ----------------------------------------------------------------------------
# sizes (section "Dequantise weights during matrix multiplication")
# ----------------------------------------------------------------------------
def bits_per_weight(group_size: int = GROUP, code_bits: int = 4, param_bits: int = 16) -> float:
    """Storage cost of one weight: its code plus its share of one scale and one bias."""
    return code_bits + 2.0 * param_bits / group_size


def checkpoint_gb(n_params: float, bits: float) -> float:
    return n_params * bits / 8.0 / 1e9

