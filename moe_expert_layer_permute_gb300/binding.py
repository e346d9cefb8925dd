"""ctypes binding of the MoE layer's C ABI (`include/moe_layer.h`).

Argument marshalling only: torch tensors become `moe_tensor` views (device pointer, dtype,
shape, strides), the current torch CUDA stream becomes the `stream` argument, and every step of
the layer runs in the CUDA library.  The library is loaded on import; if it has not been built,
importing this module raises (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

# ---- C structures ---------------------------------------------------------------------------
MOE_BF16, MOE_MXFP8, MOE_FP8_BWD, MOE_FP8_FP4 = 0, 1, 2, 3
MOE_DT_BF16, MOE_DT_F32, MOE_DT_I32 = 0, 1, 2
MOE_FLAG_SAVE_GU, MOE_FLAG_REUSE_FWD, MOE_FLAG_REUSE_WEIGHTS, MOE_FLAG_FUSED_COMBINE = 0x1, 0x2, 0x4, 0x8
(MOE_VIEW_COUNTS, MOE_VIEW_OFFSETS, MOE_VIEW_PERM, MOE_VIEW_INV, MOE_VIEW_PAD_OFFSETS, MOE_VIEW_XPERM,
 MOE_VIEW_HID, MOE_VIEW_GU, MOE_VIEW_YPART, MOE_VIEW_DG, MOE_VIEW_HW, MOE_VIEW_DYPERM) = range(12)
MOE_DEV_OK, MOE_DEV_BAD_EXPERT, MOE_DEV_TIMEOUT = 0, 1, 2
MOE_TEST_WITHHOLD_LOADS = 0x1
MX_VIEWS = {name: 32 + i for i, name in enumerate(
    ["x_r", "x_r_sf", "x_c", "x_c_sf", "h_r", "h_r_sf", "dy_r", "dy_r_sf", "dy_c", "dy_c_sf", "dg_r", "dg_r_sf",
     "dg_c", "dg_c_sf", "hw_c", "hw_c_sf", "w13_r", "w13_r_sf", "w13_c", "w13_c_sf", "w2_r", "w2_r_sf", "w2_c",
     "w2_c_sf"])}
ERRORS = {0: "MOE_OK", -1: "MOE_ERR_NULL", -2: "MOE_ERR_SHAPE", -3: "MOE_ERR_DTYPE", -4: "MOE_ERR_LAYOUT",
          -5: "MOE_ERR_ALIGN", -6: "MOE_ERR_SCRATCH", -7: "MOE_ERR_STATE", -8: "MOE_ERR_UNSUPPORTED",
          -9: "MOE_ERR_CUDA", -10: "MOE_ERR_DEVICE"}
ERR = {v: k for k, v in ERRORS.items()}

# every symbol the header declares
EXPORTS = ("moe_scratch_bytes", "moe_fwd", "moe_bwd", "moe_read_device_status", "moe_strerror",
           "moe_scratch_view", "moe_trace_enable", "moe_trace_reset", "moe_trace_read", "moe_route_static",
           "moe_router_fwd", "moe_router_bwd", "moe_set_wait_limit")


class MoeTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 3), ("stride", ctypes.c_int64 * 3)]


class MoeDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64), ("E", ctypes.c_int64),
                ("k", ctypes.c_int64), ("precision", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class MoeScratch(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("bytes", ctypes.c_uint64), ("desc", MoeDesc),
                ("epoch", ctypes.c_uint64), ("state", ctypes.c_uint64 * 4)]


_P = ctypes.POINTER


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built ({path}); run moe_expert_layer_permute_gb300.build.build()")
    lib = ctypes.CDLL(path)
    lib.moe_scratch_bytes.argtypes = [_P(MoeDesc)]
    lib.moe_scratch_bytes.restype = ctypes.c_size_t
    lib.moe_fwd.argtypes = [_P(MoeTensor)] * 6 + [_P(MoeScratch), ctypes.c_void_p]
    lib.moe_fwd.restype = ctypes.c_int
    lib.moe_bwd.argtypes = [_P(MoeTensor)] * 10 + [_P(MoeScratch), ctypes.c_void_p]
    lib.moe_bwd.restype = ctypes.c_int
    lib.moe_read_device_status.argtypes = [_P(MoeScratch), ctypes.c_void_p, _P(ctypes.c_int)]
    lib.moe_read_device_status.restype = ctypes.c_int
    lib.moe_strerror.argtypes = [ctypes.c_int]
    lib.moe_strerror.restype = ctypes.c_char_p
    lib.moe_scratch_view.argtypes = [_P(MoeDesc), ctypes.c_int, _P(ctypes.c_uint64), _P(ctypes.c_uint64)]
    lib.moe_scratch_view.restype = ctypes.c_int
    lib.moe_trace_enable.argtypes = [ctypes.c_int]
    lib.moe_trace_enable.restype = ctypes.c_int
    lib.moe_trace_reset.argtypes = []
    lib.moe_trace_reset.restype = ctypes.c_int
    lib.moe_trace_read.argtypes = [_P(ctypes.c_char_p), _P(ctypes.c_int64), _P(ctypes.c_double), _P(ctypes.c_int)]
    lib.moe_trace_read.restype = ctypes.c_int
    lib.moe_route_static.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64] + \
        [ctypes.c_void_p] * 5
    lib.moe_route_static.restype = ctypes.c_int
    lib.moe_router_fwd.argtypes = [_P(MoeTensor)] * 3 + [ctypes.c_void_p]
    lib.moe_router_fwd.restype = ctypes.c_int
    lib.moe_router_bwd.argtypes = [_P(MoeTensor)] * 4 + [ctypes.c_void_p]
    lib.moe_router_bwd.restype = ctypes.c_int
    lib.moe_set_wait_limit.argtypes = [_P(MoeScratch), ctypes.c_int64, ctypes.c_uint32]
    lib.moe_set_wait_limit.restype = ctypes.c_int
    return lib


LIB = _load()


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {ERRORS.get(code, code)} ({strerror(code)})")


def strerror(code: int) -> str:
    return LIB.moe_strerror(code).decode()


_DT = {torch.bfloat16: MOE_DT_BF16, torch.float32: MOE_DT_F32, torch.int32: MOE_DT_I32}


def as_moe_tensor(t: torch.Tensor) -> MoeTensor:
    m = MoeTensor()
    m.data = t.data_ptr() if t.numel() else 0
    m.dtype = _DT.get(t.dtype, -1)
    m.ndim = t.dim()
    for i in range(min(t.dim(), 3)):
        m.shape[i] = t.shape[i]
        m.stride[i] = t.stride(i)
    return m


def make_desc(T, H, I, E, k, precision=MOE_BF16, flags=0) -> MoeDesc:
    return MoeDesc(T, H, I, E, k, precision, flags)


def moe_scratch_bytes(desc: MoeDesc) -> int:
    return int(LIB.moe_scratch_bytes(ctypes.byref(desc)))


def view_span(desc: MoeDesc, which: int) -> tuple:
    """(byte offset, byte count) of a named scratch region for `desc` (moe_scratch_view)."""
    off, nbytes = ctypes.c_uint64(), ctypes.c_uint64()
    rc = LIB.moe_scratch_view(ctypes.byref(desc), which, ctypes.byref(off), ctypes.byref(nbytes))
    if rc:
        raise MoeError(rc, "moe_scratch_view")
    return off.value, nbytes.value


class Scratch:
    """A caller-owned device scratch buffer (a torch uint8 tensor) and its C handle."""

    def __init__(self, T, H, I, E, k, precision=MOE_BF16, device="cuda"):
        desc = make_desc(T, H, I, E, k, precision)
        n = moe_scratch_bytes(desc)
        if n == 0:
            raise MoeError(ERR["MOE_ERR_SHAPE"], "moe_scratch_bytes")
        self.buffer = torch.zeros(n, dtype=torch.uint8, device=device)
        self.handle = MoeScratch()
        self.handle.data = self.buffer.data_ptr()
        self.handle.bytes = n
        self.handle.desc = desc

    @property
    def desc(self) -> MoeDesc:
        return self.handle.desc

    @property
    def epoch(self) -> int:
        """The caller's counter of in-place updates of x / W13 / W2 (see MOE_FLAG_REUSE_*)."""
        return int(self.handle.epoch)

    @epoch.setter
    def epoch(self, value: int) -> None:
        self.handle.epoch = value

    def set_wait_limit(self, cycles: int = 0, test_flags: int = 0) -> None:
        """Pipeline wait limit in SM cycles for later calls (0: the default) and MOE_TEST_* flags."""
        rc = LIB.moe_set_wait_limit(ctypes.byref(self.handle), cycles, test_flags)
        if rc:
            raise MoeError(rc, "moe_set_wait_limit")

    def view(self, which: int, dtype: torch.dtype, shape) -> torch.Tensor:
        off, nbytes = view_span(self.handle.desc, which)
        raw = self.buffer[off:off + nbytes]
        return raw.view(dtype).view(*shape)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def moe_fwd(x, topk_idx, topk_w, W13, W2, y, scratch: Scratch, stream=None, flags: int = 0) -> None:
    scratch.handle.desc.flags = flags
    args = [as_moe_tensor(t) for t in (x, topk_idx, topk_w, W13, W2, y)]
    rc = LIB.moe_fwd(*[ctypes.byref(a) for a in args], ctypes.byref(scratch.handle), _stream_ptr(stream))
    if rc:
        raise MoeError(rc, "moe_fwd")


def moe_bwd(dy, x, topk_idx, topk_w, W13, W2, dx, dW13, dW2, dtopk_w, scratch: Scratch, stream=None,
            flags: int = 0) -> None:
    scratch.handle.desc.flags = flags
    args = [as_moe_tensor(t) for t in (dy, x, topk_idx, topk_w, W13, W2, dx, dW13, dW2, dtopk_w)]
    rc = LIB.moe_bwd(*[ctypes.byref(a) for a in args], ctypes.byref(scratch.handle), _stream_ptr(stream))
    if rc:
        raise MoeError(rc, "moe_bwd")


def moe_read_device_status(scratch: Scratch, stream=None) -> int:
    st = ctypes.c_int(0)
    rc = LIB.moe_read_device_status(ctypes.byref(scratch.handle), _stream_ptr(stream), ctypes.byref(st))
    if rc:
        raise MoeError(rc, "moe_read_device_status")
    return st.value


def moe_trace_enable(on: bool) -> None:
    LIB.moe_trace_enable(1 if on else 0)


def moe_trace_reset() -> None:
    LIB.moe_trace_reset()


def moe_trace_read() -> dict:
    """{kernel name: (launches, total ms)} of the launches recorded since the last reset."""
    cap = 64
    names = (ctypes.c_char_p * cap)()
    launches = (ctypes.c_int64 * cap)()
    ms = (ctypes.c_double * cap)()
    n = ctypes.c_int(cap)
    LIB.moe_trace_read(names, launches, ms, ctypes.byref(n))
    return {names[i].decode(): (int(launches[i]), float(ms[i])) for i in range(min(n.value, cap))}


def moe_route_static(topk_idx, E: int, counts, offsets, perm, inv, stream=None) -> None:
    """Routing bookkeeping into caller-owned int32 tensors, with no scratch buffer (the library's
    static device array instead): counts [E], offsets [E+1], perm [T*k], inv [T*k]."""
    T, k = topk_idx.shape
    for t in (topk_idx, counts, offsets, perm, inv):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise MoeError(ERR["MOE_ERR_DTYPE"], "moe_route_static")
    if counts.numel() != E or offsets.numel() != E + 1 or perm.numel() != T * k or inv.numel() != T * k:
        raise MoeError(ERR["MOE_ERR_SHAPE"], "moe_route_static")
    rc = LIB.moe_route_static(topk_idx.data_ptr(), T, k, E, counts.data_ptr(), offsets.data_ptr(),
                              perm.data_ptr(), inv.data_ptr(), _stream_ptr(stream))
    if rc:
        raise MoeError(rc, "moe_route_static")


def moe_router_fwd(logits, topk_idx, topk_w, stream=None) -> None:
    """Top-k router: logits fp32 [T, E] -> topk_idx int32 [T, k], topk_w fp32 [T, k]."""
    args = [as_moe_tensor(t) for t in (logits, topk_idx, topk_w)]
    rc = LIB.moe_router_fwd(*[ctypes.byref(a) for a in args], _stream_ptr(stream))
    if rc:
        raise MoeError(rc, "moe_router_fwd")


def moe_router_bwd(topk_idx, topk_w, dtopk_w, dlogits, stream=None) -> None:
    """Router backward: dlogits fp32 [T, E] from the weights' gradient dtopk_w fp32 [T, k]."""
    args = [as_moe_tensor(t) for t in (topk_idx, topk_w, dtopk_w, dlogits)]
    rc = LIB.moe_router_bwd(*[ctypes.byref(a) for a in args], _stream_ptr(stream))
    if rc:
        raise MoeError(rc, "moe_router_bwd")
