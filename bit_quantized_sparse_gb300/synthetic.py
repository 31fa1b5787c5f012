"""Seeded synthetic inputs for the W4 group-affine sparse-MoE layer.

This module draws layers and token batches with the shapes and value
distributions of the layer described in "Optimizing on-device inference for
Apple Silicon" (section "Qwen creates three different workload shapes": 256
experts, top-8, one shared expert; section "Dequantise weights during matrix
multiplication": 4-bit codes, one bf16 scale and one bf16 bias per 64
weights).  It implements none of the layer's arithmetic: no dequantisation,
no top-k selection, no softmax, no expert projection.  The only arithmetic on
drawn values is the input screen in `draw_tokens`, which recomputes the raw
router scores x.W_r (+bias) in float64 solely to redraw tokens whose leading
scores are closer than the required margin.

Everything is numpy (PCG64) so the same seed gives the same bytes on any host.

Layout of a drawn layer (all numpy, C-contiguous):
  * gate/up codes   uint32 [E][I][H/8]   (row = output feature, words along input)
  * down codes      uint32 [E][H][I/8]
  * scales/biases   uint16 bf16 bit patterns [E][rows][cols/64]
  * shared expert   same without the leading E
  * router_w        float32 [H][E]; router_bias float32 [E] or None
  * shared_gate     float32 [H]
Eight 4-bit codes sit in each uint32, the lowest-index column in the lowest
nibble.  The format variants (code_bits = 8, unsigned or FP8 E4M3 codes) hold
four one-byte codes per uint32, the lowest-index column in the lowest byte, so
their codes arrays are [..][rows][cols/4].
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GROUP = 64          # weights sharing one scale and one bias
MARGIN = 1e-2       # minimum gap between adjacent leading router scores
CODES_UINT = 0      # code_format: unsigned integer codes (4 or 8 bits)
CODES_E4M3 = 1      # code_format: FP8 E4M3 codes (8 bits)

# Workload table.  Each entry is a layer shape plus a batch description.
CONFIGS = {
    # tiny layer the oracle finishes in well under a second
    "tiny_T4": dict(T=4, H=256, E=16, top_k=2, I=128, zipf=None, seed=0),
    # batch-1 decode step on the full layer, uniform expert popularity
    "decode_T1": dict(T=1, H=2048, E=256, top_k=8, I=512, zipf=None, seed=1),
    # short prefill, Zipf(1.0)-skewed routing
    "prefill_T512": dict(T=512, H=2048, E=256, top_k=8, I=512, zipf=1.0, seed=2),
    # 4K-token prefill, Zipf(1.0)-skewed routing
    "prefill_T4096": dict(T=4096, H=2048, E=256, top_k=8, I=512, zipf=1.0, seed=3),
    # 16K-token prefill in four 4096-row chunks, then 64 batch-1 decode steps,
    # Zipf(1.2)-skewed routing
    "long_T16384": dict(T=16384, H=2048, E=256, top_k=8, I=512, zipf=1.2, seed=4,
                        chunk=4096, decode_steps=64),
    # the 8-bit affine weight-format variant of the full layer, short prefill
    "w8_T512": dict(T=512, H=2048, E=256, top_k=8, I=512, zipf=1.0, seed=5, bits=8),
    # the 8-bit variant of the tiny layer
    "w8_tiny_T4": dict(T=4, H=256, E=16, top_k=2, I=128, zipf=None, seed=6, bits=8),
    # FP8 E4M3 codes (one byte per weight, four per word) with the same group
    # scale and bias, full layer and tiny layer
    "e4m3_T512": dict(T=512, H=2048, E=256, top_k=8, I=512, zipf=1.0, seed=7, bits=8, fmt=CODES_E4M3),
    "e4m3_tiny_T4": dict(T=4, H=256, E=16, top_k=2, I=128, zipf=None, seed=8, bits=8, fmt=CODES_E4M3),
}


@dataclasses.dataclass
class W4Matrix:
    """One group-affine 4-bit matrix (or a stack of them along a leading E axis)."""
    codes: np.ndarray      # uint32 [..., rows, cols/8]
    scales: np.ndarray     # uint16 bf16 bits [..., rows, cols/64]
    biases: np.ndarray     # uint16 bf16 bits [..., rows, cols/64]


@dataclasses.dataclass
class W4Layer:
    H: int
    E: int
    I: int
    top_k: int
    router_w: np.ndarray               # float32 [H][E]
    router_bias: Optional[np.ndarray]  # float32 [E] or None
    shared_gate: np.ndarray            # float32 [H]
    gate: W4Matrix                     # [E][I][H/8]
    up: W4Matrix                       # [E][I][H/8]
    down: W4Matrix                     # [E][H][I/8]
    sh_gate: W4Matrix                  # [I][H/8]
    sh_up: W4Matrix                    # [I][H/8]
    sh_down: W4Matrix                  # [H][I/8]
    code_bits: int = 4                 # 4 (eight codes per word) or 8 (four codes per word)
    code_format: int = CODES_UINT      # CODES_UINT or CODES_E4M3 (8-bit codes only)

    def nbytes_expert(self) -> int:
        """Bytes of one expert's three matrices (codes + scales + biases)."""
        w = 3 * self.H * self.I
        return w * self.code_bits // 8 + 2 * 2 * (w // GROUP)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def _e4m3_bytes(sign, expo, mant):
    """Assemble FP8 E4M3 bit patterns from their fields: sign << 7 | exponent
    field << 3 | mantissa field (bit packing only; no value is computed)."""
    return (sign << 7) | (expo << 3) | mant


def _draw_matrix(rng: np.random.Generator, lead: tuple, rows: int, cols: int, bits: int = 4,
                 fmt: int = CODES_UINT) -> W4Matrix:
    """4 bits: codes uniform in [0,15] (a uniform 32-bit word is eight uniform
    nibbles); s = bf16(|N(0,0.02)|); b = bf16(-8 s + N(0,0.002)).  8 bits: codes
    uniform in [0,255], s = bf16(|N(0,0.02)| / 17), b = bf16(-128 s + N(0,0.002)),
    so that the weights have about the same spread as the 4-bit ones.  FP8 E4M3:
    each byte has a uniform sign, an exponent field uniform in [3,10] and a
    uniform mantissa field (magnitudes 2^-4 .. 15, never NaN; their rms is about
    that of the centred 4-bit codes); s = bf16(|N(0,0.02)|), b = bf16(N(0,0.002))."""
    assert cols % GROUP == 0 and bits in (4, 8) and (fmt == CODES_UINT or bits == 8)
    shape_g = lead + (rows, cols // GROUP)
    if fmt == CODES_E4M3:
        shape_b = lead + (rows, cols // 4, 4)
        byt = _e4m3_bytes(rng.integers(0, 2, size=shape_b, dtype=np.uint32),
                          rng.integers(3, 11, size=shape_b, dtype=np.uint32),
                          rng.integers(0, 8, size=shape_b, dtype=np.uint32))
        codes = (byt[..., 0] | (byt[..., 1] << 8) | (byt[..., 2] << 16) | (byt[..., 3] << 24)).astype(np.uint32)
        s_bits = f32_to_bf16_bits(np.abs(rng.normal(0.0, 0.02, size=shape_g)).astype(np.float32))
        b_bits = f32_to_bf16_bits(rng.normal(0.0, 0.002, size=shape_g).astype(np.float32))
        return W4Matrix(codes, s_bits, b_bits)
    codes = rng.integers(0, 1 << 32, size=lead + (rows, cols * bits // 32), dtype=np.uint32)
    div, mid = (1.0, 8.0) if bits == 4 else (17.0, 128.0)
    s_bits = f32_to_bf16_bits((np.abs(rng.normal(0.0, 0.02, size=shape_g)) / div).astype(np.float32))
    s = bf16_bits_to_f32(s_bits)
    b_bits = f32_to_bf16_bits((-mid * s + rng.normal(0.0, 0.002, size=shape_g)).astype(np.float32))
    return W4Matrix(codes, s_bits, b_bits)


def zipf_bias(E: int, s: float) -> np.ndarray:
    """Per-expert router offset -s*ln(rank), rank = e+1: multiplies expert e's
    softmax odds by a Zipf(s) popularity weight."""
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def draw_layer(H: int, E: int, I: int, top_k: int, zipf: Optional[float], seed: int, bits: int = 4,
               fmt: int = CODES_UINT) -> W4Layer:
    rw, rr, rs = _streams(seed, 3)
    gate = _draw_matrix(rw, (E,), I, H, bits, fmt)
    up = _draw_matrix(rw, (E,), I, H, bits, fmt)
    down = _draw_matrix(rw, (E,), H, I, bits, fmt)
    sh_gate = _draw_matrix(rs, (), I, H, bits, fmt)
    sh_up = _draw_matrix(rs, (), I, H, bits, fmt)
    sh_down = _draw_matrix(rs, (), H, I, bits, fmt)
    router_w = rr.normal(0.0, 0.05, size=(H, E)).astype(np.float32)
    shared_gate = rr.normal(0.0, 0.05, size=(H,)).astype(np.float32)
    bias = zipf_bias(E, zipf) if zipf else None
    return W4Layer(H, E, I, top_k, router_w, bias, shared_gate, gate, up, down,
                   sh_gate, sh_up, sh_down, bits, fmt)


def _screen_ok(x_bits: np.ndarray, layer: W4Layer, margin: float) -> np.ndarray:
    """Input screen: True for tokens whose top-(k+1) raw scores are pairwise
    separated by at least `margin` (adjacent pairs after sorting)."""
    x = bf16_bits_to_f32(x_bits).astype(np.float64)
    sc = x @ layer.router_w.astype(np.float64)
    if layer.router_bias is not None:
        sc = sc + layer.router_bias.astype(np.float64)
    kk = min(layer.top_k + 1, layer.E)
    lead = -np.sort(-sc, axis=1)[:, :kk]
    if kk < 2:
        return np.ones(x.shape[0], dtype=bool)
    return np.all(lead[:, :-1] - lead[:, 1:] >= margin, axis=1)


def draw_tokens(layer: W4Layer, T: int, seed: int, stream: int = 0,
                margin: Optional[float] = MARGIN) -> np.ndarray:
    """x = bf16(N(0,1)) of shape [T][H] (bf16 bits).  With a margin, any token
    failing the score screen is redrawn from the same stream until it passes."""
    rng = _streams(seed * 1000003 + 17 + stream, 1)[0]
    x = f32_to_bf16_bits(rng.normal(0.0, 1.0, size=(T, layer.H)).astype(np.float32))
    if margin is None or T == 0:
        return x
    for _ in range(1000):
        bad = np.nonzero(~_screen_ok(x, layer, margin))[0]
        if bad.size == 0:
            return x
        x[bad] = f32_to_bf16_bits(rng.normal(0.0, 1.0, size=(bad.size, layer.H)).astype(np.float32))
    raise RuntimeError("input screen did not converge")


def draw_config(name: str, T: Optional[int] = None, stream: int = 0):
    """Layer and token batch of a named workload; T overrides the batch size."""
    c = CONFIGS[name]
    layer = draw_layer(c["H"], c["E"], c["I"], c["top_k"], c["zipf"], c["seed"], c.get("bits", 4),
                       c.get("fmt", CODES_UINT))
    x = draw_tokens(layer, c["T"] if T is None else T, c["seed"], stream)
    return layer, x


def draw_layer_torch(H: int, E: int, I: int, top_k: int, zipf: Optional[float], seed: int, device="cuda",
                     bits: int = 4, fmt: int = CODES_UINT):
    """Same recipe as draw_layer, drawn directly on a device with a seeded torch
    generator (fast enough for many layer replicas; the values differ from the
    numpy draw of the same seed).  Returns a W4Layer whose arrays are torch
    tensors: codes int32 (bit patterns of the uint32 words), scales/biases
    int16 (bf16 bit patterns), router float32."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))

    div, mid = (1.0, 8.0) if bits == 4 else (17.0, 128.0)

    def mat(lead, rows, cols):
        shape_g = lead + (rows, cols // GROUP)
        if fmt == CODES_E4M3:
            shape_b = lead + (rows, cols // 4, 4)
            byt = _e4m3_bytes(torch.randint(0, 2, shape_b, generator=g, device=device, dtype=torch.int64),
                              torch.randint(3, 11, shape_b, generator=g, device=device, dtype=torch.int64),
                              torch.randint(0, 8, shape_b, generator=g, device=device, dtype=torch.int64))
            codes = (byt[..., 0] | (byt[..., 1] << 8) | (byt[..., 2] << 16) | (byt[..., 3] << 24))
            codes = torch.where(codes >= (1 << 31), codes - (1 << 32), codes).to(torch.int32)
            s = (torch.randn(shape_g, generator=g, device=device) * 0.02).abs().to(torch.bfloat16)
            b = (torch.randn(shape_g, generator=g, device=device) * 0.002).to(torch.bfloat16)
            return W4Matrix(codes, s.view(torch.int16), b.view(torch.int16))
        codes = torch.randint(-(1 << 31), 1 << 31, lead + (rows, cols * bits // 32), generator=g, device=device,
                              dtype=torch.int64).to(torch.int32)
        s = ((torch.randn(shape_g, generator=g, device=device) * 0.02).abs() / div).to(torch.bfloat16)
        b = (-mid * s.float() + torch.randn(shape_g, generator=g, device=device) * 0.002).to(torch.bfloat16)
        return W4Matrix(codes, s.view(torch.int16), b.view(torch.int16))

    gate, up, down = mat((E,), I, H), mat((E,), I, H), mat((E,), H, I)
    sh_gate, sh_up, sh_down = mat((), I, H), mat((), I, H), mat((), H, I)
    router_w = torch.randn((H, E), generator=g, device=device) * 0.05
    shared_gate = torch.randn((H,), generator=g, device=device) * 0.05
    bias = torch.from_numpy(zipf_bias(E, zipf)).to(device) if zipf else None
    return W4Layer(H, E, I, top_k, router_w, bias, shared_gate, gate, up, down, sh_gate, sh_up, sh_down, bits,
                   fmt)
