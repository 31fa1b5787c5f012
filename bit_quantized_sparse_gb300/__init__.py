"""GB300-native W4 group-affine sparse-MoE layer.

The compute path is the CUDA library `libmoe_w4.so` (sources in `csrc/`,
C header `include/moe_w4.h`); `moe_w4` is its thin ctypes binding and raises
at import if the library has not been built.  `synthetic` draws seeded
inputs.
"""
__all__ = ["moe_w4", "synthetic"]
