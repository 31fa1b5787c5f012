"""Thin ctypes binding of libmoe_w4.so (C header include/moe_w4.h).

Argument marshalling only: every step of the layer runs in the CUDA library.
Importing this module raises ImportError if the library has not been built
(`python -m bit_quantized_sparse_gb300._build`); there is no fallback.

Two levels:
  * the C entry points under their own names (moe_w4_route,
    moe_w4_forward_decode, moe_w4_forward_prefill, moe_w4_workspace_size,
    moe_w4_workspace_init, moe_w4_status_offset, moe_w4_strerror), taking raw
    device pointers (ints), a MoeW4Layer struct and a stream handle;
  * `DeviceLayer`, which keeps a layer's tensors on the GPU, and `route`,
    `forward_decode`, `forward_prefill`, which take torch tensors, allocate
    outputs with torch and raise MoeW4Error on a non-zero status.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# MOE_W4_DEBUG=1 selects the build with device-side bounds checks (and host-side
# error messages on stderr); build it with `python -m bit_quantized_sparse_gb300._build --debug`
DEBUG = os.environ.get("MOE_W4_DEBUG", "") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libmoe_w4_debug.so" if DEBUG else "libmoe_w4.so")
if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -m bit_quantized_sparse_gb300._build"
                      f"{' --debug' if DEBUG else ''}`")
_lib = ctypes.CDLL(LIB_PATH)

c_int, c_size_t, c_void_p, c_char_p = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p

MOE_W4_OK = 0
MOE_W4_ERR_INVALID = -1
MOE_W4_ERR_UNSUPPORTED = -2
MOE_W4_ERR_WORKSPACE = -3
MOE_W4_ERR_LAUNCH = -4
MOE_W4_ERR_DEVICE = -5
MOE_W4_ERR_ALIGN = -6
MOE_W4_ERR_SCRATCH = -7
MOE_W4_CODES_UINT = 0
MOE_W4_CODES_E4M3 = 1
MOE_W4_ABLATE_HOST_ROUTING = 1       # include/moe_w4_ablation.h
MOE_W4_ABLATE_SEPARATE_DEQUANT = 2
# bits of the device status word (include/moe_w4.h)
MOE_W4_STATUS_WAIT_TIMEOUT = 1
MOE_W4_STATUS_BAD_INDEX = 2
MOE_W4_STATUS_FP16_RANGE = 4
DECODE_MAX_T = 16
MAX_TOKENS = 1 << 22                 # MOE_W4_MAX_TOKENS
MOE_W4_PATH_FUSED_ROWS = 1           # moe_w4_decode_path
MOE_W4_PATH_GROUPED = 2


class MoeW4Mat(ctypes.Structure):
    _fields_ = [("codes", c_void_p), ("scales", c_void_p), ("biases", c_void_p)]


class MoeW4Layer(ctypes.Structure):
    _fields_ = [("H", c_int), ("E", c_int), ("I", c_int), ("top_k", c_int),
                ("router_w", c_void_p), ("router_bias", c_void_p), ("shared_gate", c_void_p),
                ("gate", MoeW4Mat), ("up", MoeW4Mat), ("down", MoeW4Mat),
                ("sh_gate", MoeW4Mat), ("sh_up", MoeW4Mat), ("sh_down", MoeW4Mat), ("code_bits", c_int),
                ("code_format", c_int), ("router_prep", c_void_p)]


_P = ctypes.POINTER(MoeW4Layer)
_SIGS = {
    "moe_w4_workspace_size": (c_size_t, [_P, c_int]),
    "moe_w4_router_prep_bytes": (c_size_t, [_P]),
    "moe_w4_prepare_router": (c_int, [_P, c_void_p, c_size_t, c_void_p]),
    "moe_w4_workspace_init": (c_int, [c_void_p, c_size_t, c_void_p]),
    "moe_w4_status_offset": (c_size_t, []),
    "moe_w4_route": (c_int, [_P, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_w4_forward_decode": (c_int, [_P, c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_w4_forward_prefill": (c_int, [_P, c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "moe_w4_ablation_prefill": (c_int, [_P, c_int, c_void_p, c_void_p, c_void_p, c_size_t, c_int, c_void_p,
                                        c_size_t, c_void_p]),
    "moe_w4_ablation_scratch_bytes": (c_size_t, [_P, c_int]),
    "moe_w4_set_trace_events": (c_int, [c_void_p, c_int]),
    "moe_w4_set_tile_override": (c_int, [c_int, c_int]),
    "moe_w4_set_decode_fused_rows": (c_int, [c_int]),
    "moe_w4_decode_path": (c_int, [_P, c_int, ctypes.POINTER(c_int)]),
    "moe_w4_test_refuse_fused_after": (c_int, [c_int]),
    "moe_w4_last_traced_kernels": (c_int, []),
    "moe_w4_forward_decode_noalloc": (c_int, [_P, c_int, c_void_p, c_void_p, c_void_p]),
    "moe_w4_noalloc_status": (c_int, [c_void_p, c_void_p]),
    "moe_w4_noalloc_test_skip_publish": (c_int, [c_int]),
    "moe_w4_test_skip_publish": (c_int, [c_void_p, c_size_t, c_int, c_void_p]),
    "moe_w4_test_block_records_bytes": (c_size_t, [_P, c_int]),
    "moe_w4_test_block_records": (c_int, [_P, c_int, c_void_p, c_size_t, c_void_p, c_size_t, c_void_p]),
    "moe_w4_strerror": (c_char_p, [c_int]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype, _f.argtypes = _res, _args

EXPORTED = tuple(_SIGS)

moe_w4_workspace_size = _lib.moe_w4_workspace_size
moe_w4_router_prep_bytes = _lib.moe_w4_router_prep_bytes
moe_w4_prepare_router = _lib.moe_w4_prepare_router
moe_w4_workspace_init = _lib.moe_w4_workspace_init
moe_w4_status_offset = _lib.moe_w4_status_offset
moe_w4_route = _lib.moe_w4_route
moe_w4_forward_decode = _lib.moe_w4_forward_decode
moe_w4_forward_prefill = _lib.moe_w4_forward_prefill
moe_w4_ablation_prefill = _lib.moe_w4_ablation_prefill
moe_w4_ablation_scratch_bytes = _lib.moe_w4_ablation_scratch_bytes
moe_w4_set_trace_events = _lib.moe_w4_set_trace_events
moe_w4_set_tile_override = _lib.moe_w4_set_tile_override
moe_w4_set_decode_fused_rows = _lib.moe_w4_set_decode_fused_rows
moe_w4_decode_path = _lib.moe_w4_decode_path
moe_w4_test_refuse_fused_after = _lib.moe_w4_test_refuse_fused_after
moe_w4_last_traced_kernels = _lib.moe_w4_last_traced_kernels
moe_w4_forward_decode_noalloc = _lib.moe_w4_forward_decode_noalloc
moe_w4_noalloc_status = _lib.moe_w4_noalloc_status
moe_w4_noalloc_test_skip_publish = _lib.moe_w4_noalloc_test_skip_publish
moe_w4_test_skip_publish = _lib.moe_w4_test_skip_publish
moe_w4_test_block_records_bytes = _lib.moe_w4_test_block_records_bytes
moe_w4_test_block_records = _lib.moe_w4_test_block_records


def moe_w4_strerror(status: int) -> str:
    return _lib.moe_w4_strerror(status).decode()


class MoeW4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {moe_w4_strerror(status)} ({status})")
        self.status = status


def _check(status: int, where: str):
    if status != MOE_W4_OK:
        raise MoeW4Error(status, where)


# ---------------------------------------------------------------------------
# torch-level helpers
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class DeviceLayer:
    """A layer's tensors resident on one GPU plus the C struct pointing at them.

    Build it from any object with the attributes of synthetic.W4Layer (numpy
    arrays: uint32 codes, uint16 bf16 bit patterns, float32 router)."""

    def __init__(self, layer, device="cuda", prepare_router=True):
        torch = _torch()
        self.H, self.E, self.I, self.top_k = int(layer.H), int(layer.E), int(layer.I), int(layer.top_k)
        self.device = torch.device(device)

        tdt = {np.int32: torch.int32, np.int16: torch.int16, np.float32: torch.float32}

        def dev(a, dt):
            if torch.is_tensor(a):
                return a.to(self.device).contiguous().view(tdt[dt])
            return torch.from_numpy(np.ascontiguousarray(a).view(dt)).to(self.device)

        def mat(m):
            return (dev(m.codes, np.int32), dev(m.scales, np.int16), dev(m.biases, np.int16))

        self.router_w = dev(layer.router_w, np.float32)
        self.router_bias = None if layer.router_bias is None else dev(layer.router_bias, np.float32)
        self.shared_gate = dev(layer.shared_gate, np.float32)
        self.mats = {n: mat(getattr(layer, n)) for n in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")}
        self.c = MoeW4Layer()
        self.c.H, self.c.E, self.c.I, self.c.top_k = self.H, self.E, self.I, self.top_k
        self.code_bits = int(getattr(layer, "code_bits", 4))
        self.c.code_bits = self.code_bits
        self.code_format = int(getattr(layer, "code_format", MOE_W4_CODES_UINT))
        self.c.code_format = self.code_format
        self.c.router_w = _ptr(self.router_w)
        self.c.router_bias = _ptr(self.router_bias)
        self.c.shared_gate = _ptr(self.shared_gate)
        for n, (c, s, b) in self.mats.items():
            setattr(self.c, n, MoeW4Mat(c.data_ptr(), s.data_ptr(), b.data_ptr()))
        # the router weights split once for the tensor-core routing (none for a
        # layer the library rejects: its calls return the error instead)
        self.router_prep = None
        nprep = moe_w4_router_prep_bytes(ctypes.byref(self.c)) if prepare_router else 0
        if nprep:
            self.router_prep = torch.empty(nprep, dtype=torch.uint8, device=self.device)
            _check(moe_w4_prepare_router(ctypes.byref(self.c), self.router_prep.data_ptr(), nprep, _stream()),
                   "prepare_router")
            self.c.router_prep = self.router_prep.data_ptr()
        self._ws = None
        self._ws_T = -1

    def workspace_size(self, T_max: int) -> int:
        return moe_w4_workspace_size(ctypes.byref(self.c), T_max)

    def workspace(self, T_max: int):
        """A zero-initialised workspace for calls with up to T_max tokens (cached)."""
        torch = _torch()
        if self._ws is None or self._ws_T < T_max:
            n = self.workspace_size(T_max)
            if n == 0:
                raise MoeW4Error(MOE_W4_ERR_UNSUPPORTED, "workspace_size")
            self._ws = torch.empty(n, dtype=torch.uint8, device=self.device)
            self._ws_T = T_max
            _check(moe_w4_workspace_init(self._ws.data_ptr(), n, _stream()), "workspace_init")
        return self._ws

    def status(self) -> int:
        """Device status word of the cached workspace (synchronises)."""
        torch = _torch()
        if self._ws is None:
            return 0
        off = moe_w4_status_offset()
        return int(self._ws[off:off + 4].view(torch.int32).item())


def route(layer: DeviceLayer, x, stream=None):
    """Routing outputs of moe_w4_route as a dict of device tensors."""
    torch = _torch()
    T = int(x.shape[0])
    dev = layer.device
    k, E = layer.top_k, layer.E
    o = dict(topk_idx=torch.empty((T, k), dtype=torch.int32, device=dev),
             topk_w=torch.empty((T, k), dtype=torch.float32, device=dev),
             gamma=torch.empty((T,), dtype=torch.float32, device=dev),
             counts=torch.empty((E,), dtype=torch.int32, device=dev),
             offsets=torch.empty((E + 1,), dtype=torch.int32, device=dev),
             perm=torch.empty((T * k,), dtype=torch.int32, device=dev),
             inv=torch.empty((T * k,), dtype=torch.int32, device=dev))
    ws = layer.workspace(T)
    _check(moe_w4_route(ctypes.byref(layer.c), T, _ptr(x), *[o[n].data_ptr() for n in
                        ("topk_idx", "topk_w", "gamma", "counts", "offsets", "perm", "inv")],
                        ws.data_ptr(), ws.numel(), _stream(stream)), "moe_w4_route")
    return o


def forward_decode(layer: DeviceLayer, x, out=None, stream=None):
    torch = _torch()
    T = int(x.shape[0])
    if out is None:
        out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=layer.device)
    ws = layer.workspace(T)
    _check(moe_w4_forward_decode(ctypes.byref(layer.c), T, _ptr(x), _ptr(out), ws.data_ptr(), ws.numel(),
                                 _stream(stream)), "moe_w4_forward_decode")
    return out


def decode_path(layer: DeviceLayer, T: int) -> int:
    """MOE_W4_PATH_FUSED_ROWS or MOE_W4_PATH_GROUPED: the path moe_w4_forward_decode takes for T rows."""
    p = c_int(0)
    _check(moe_w4_decode_path(ctypes.byref(layer.c), int(T), ctypes.byref(p)), "moe_w4_decode_path")
    return p.value


def forward_prefill(layer: DeviceLayer, x, out=None, stream=None, ws=None):
    torch = _torch()
    T = int(x.shape[0])
    if out is None:
        out = torch.empty((T, layer.H), dtype=torch.bfloat16, device=layer.device)
    if ws is None:
        ws = layer.workspace(T)
    _check(moe_w4_forward_prefill(ctypes.byref(layer.c), T, _ptr(x), _ptr(out), ws.data_ptr(), ws.numel(),
                                  _stream(stream)), "moe_w4_forward_prefill")
    return out


def tokens_to_device(x_bits: np.ndarray, device="cuda"):
    """bf16 bit patterns [T][H] (uint16) -> torch.bfloat16 tensor on `device`."""
    torch = _torch()
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).to(device).view(torch.bfloat16)
