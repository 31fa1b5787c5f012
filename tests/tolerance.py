"""Float tolerance of the layer output, shared by the GPU parity tests.

Stated bar: max|err| <= 2e-2 * rms(ref) and relative L2 error <= 5e-3, ref
being the float64 oracle.  The output format is bf16, as the pages require
("Optimizing on-device inference for Apple Silicon", section "Dequantise
weights during matrix multiplication": fp32 accumulation, bf16 output).  A bf16
value can sit up to half a unit in the last place (2^-8 of the value) from the
exact result, and on these workloads outputs reach about 9 rms, so even the
exact result rounded to bf16 breaks the literal max bound (see
test_tolerance_reading).  Reading taken: the max bound applies to the error
beyond that final rounding,
    max(|got - ref| - halfulp_bf16(ref)) <= 2e-2 * rms(ref),
and the relative L2 bound applies as stated.
"""
import numpy as np

MAX_REL = 2e-2
L2_REL = 5e-3


def halfulp_bf16(v):
    """Half the bf16 spacing at |v|: 2^(floor(log2|v|) - 8)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def metrics(got, ref):
    err = np.asarray(got, np.float64) - ref
    rms = np.sqrt(np.mean(ref ** 2))
    return dict(max_rel_literal=float(np.max(np.abs(err)) / rms),
                max_rel=float(np.max(np.abs(err) - halfulp_bf16(ref)) / rms),
                l2=float(np.linalg.norm(err) / np.linalg.norm(ref)))


def within(m):
    return m["max_rel"] <= MAX_REL and m["l2"] <= L2_REL
