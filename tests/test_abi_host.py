"""Host-side checks of the C ABI (no GPU needed): the library builds and loads, exports every
function `include/moe_layer.h` declares, sizes its scratch, and rejects bad arguments with the
documented status codes before anything is launched."""
import ctypes
import os
import re

import pytest
import torch

from moe_expert_layer_permute_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bd():
    build.build()
    from moe_expert_layer_permute_gb300 import binding
    return binding


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_layer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_function(bd):
    declared = _declared_functions()
    assert len(declared) >= 9
    for name in declared:
        assert hasattr(bd.LIB, name), name
        ctypes.cast(getattr(bd.LIB, name), ctypes.c_void_p)
    assert sorted(bd.EXPORTS) == declared


def test_scratch_bytes_rules(bd):
    ok = bd.make_desc(16384, 2048, 768, 128, 8)
    n = bd.moe_scratch_bytes(ok)
    assert n > 0
    n2 = bd.moe_scratch_bytes(bd.make_desc(32768, 2048, 768, 128, 8))
    assert n2 > n
    for bad in [(16, 2000, 768, 8, 2), (16, 2048, 700, 8, 2), (16, 256, 128, 4, 5), (16, 256, 128, 2000, 2),
                (-1, 256, 128, 8, 2), (16, 256, 128, 8, 0)]:
        assert bd.moe_scratch_bytes(bd.make_desc(*bad)) == 0, bad
    assert bd.moe_scratch_bytes(bd.make_desc(0, 256, 128, 8, 2)) > 0


def test_scratch_views_are_disjoint_and_aligned(bd):
    d = bd.make_desc(1000, 512, 256, 16, 4)
    total = bd.moe_scratch_bytes(d)
    spans = {}
    for v in range(12):
        off, nb = ctypes.c_uint64(), ctypes.c_uint64()
        assert bd.LIB.moe_scratch_view(ctypes.byref(d), v, ctypes.byref(off), ctypes.byref(nb)) == 0
        assert off.value % 256 == 0 and off.value + nb.value <= total
        spans[v] = (off.value, off.value + nb.value)
    # w h: the backward reads the rows the forward's gate/up epilogue stored, one region
    assert spans.pop(bd.MOE_VIEW_HW) == spans[bd.MOE_VIEW_HID]
    spans = sorted(spans.values())
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 <= b0
    off, nb = ctypes.c_uint64(), ctypes.c_uint64()
    assert bd.LIB.moe_scratch_view(ctypes.byref(d), 99, ctypes.byref(off), ctypes.byref(nb)) == bd.ERR["MOE_ERR_SHAPE"]


class _Fake:
    """moe_tensor views with fake (never dereferenced) aligned device addresses."""

    def __init__(self, bd):
        self.bd = bd
        self.addr = 1 << 20

    def t(self, shape, dt, contiguous=True, misalign=0):
        m = self.bd.MoeTensor()
        m.data = self.addr + misalign
        self.addr += 1 << 24
        m.dtype = dt
        m.ndim = len(shape)
        st = 1
        strides = []
        for s in reversed(shape):
            strides.append(st)
            st *= s
        strides = list(reversed(strides))
        if not contiguous:
            strides[0] *= 2
        for i, (s, r) in enumerate(zip(shape, strides)):
            m.shape[i] = s
            m.stride[i] = r
        return m


def _fwd_args(bd, T=256, H=256, I=128, E=8, k=2, **over):
    f = _Fake(bd)
    a = {"x": f.t((T, H), bd.MOE_DT_BF16), "idx": f.t((T, k), bd.MOE_DT_I32), "w": f.t((T, k), bd.MOE_DT_F32),
         "W13": f.t((E, 2 * I, H), bd.MOE_DT_BF16), "W2": f.t((E, H, I), bd.MOE_DT_BF16),
         "y": f.t((T, H), bd.MOE_DT_BF16)}
    a.update({k_: v(f) for k_, v in over.items()})
    s = bd.MoeScratch()
    s.desc = bd.make_desc(T, H, I, E, k)
    s.bytes = bd.moe_scratch_bytes(s.desc)
    s.data = 1 << 40
    return a, s


def _call_fwd(bd, a, s):
    return bd.LIB.moe_fwd(*[ctypes.byref(a[n]) for n in ("x", "idx", "w", "W13", "W2", "y")], ctypes.byref(s), None)


@pytest.mark.parametrize("over,code", [
    ({"x": lambda f: f.t((256, 512), 0)}, "MOE_ERR_SHAPE"),
    ({"idx": lambda f: f.t((256, 2), 1)}, "MOE_ERR_DTYPE"),
    ({"w": lambda f: f.t((256, 2), 0)}, "MOE_ERR_DTYPE"),
    ({"W13": lambda f: f.t((8, 256, 256), 0, contiguous=False)}, "MOE_ERR_LAYOUT"),
    ({"y": lambda f: f.t((256, 256), 0, misalign=8)}, "MOE_ERR_ALIGN"),
    ({"W2": lambda f: f.t((8, 128, 256), 0)}, "MOE_ERR_SHAPE"),
])
def test_fwd_rejects_bad_tensors(bd, over, code):
    a, s = _fwd_args(bd, **over)
    assert _call_fwd(bd, a, s) == bd.ERR[code]


def test_fwd_rejects_bad_scratch_and_desc(bd):
    a, s = _fwd_args(bd)
    s.bytes -= 1
    assert _call_fwd(bd, a, s) == bd.ERR["MOE_ERR_SCRATCH"]
    a, s = _fwd_args(bd)
    s.data = (1 << 40) + 64
    assert _call_fwd(bd, a, s) == bd.ERR["MOE_ERR_SCRATCH"]
    a, s = _fwd_args(bd)
    s.desc.H = 384
    assert _call_fwd(bd, a, s) == bd.ERR["MOE_ERR_SHAPE"]
    a, s = _fwd_args(bd)
    s.desc.precision = 7
    assert _call_fwd(bd, a, s) == bd.ERR["MOE_ERR_UNSUPPORTED"]
    assert bd.LIB.moe_fwd(None, None, None, None, None, None, None, None) == bd.ERR["MOE_ERR_NULL"]


def test_bwd_reuse_needs_a_saved_forward(bd):
    a, s = _fwd_args(bd)
    f = _Fake(bd)
    f.addr = 1 << 36
    dy = f.t((256, 256), 0); dx = f.t((256, 256), 0)
    dW13 = f.t((8, 256, 256), 1); dW2 = f.t((8, 256, 128), 1); dtw = f.t((256, 2), 1)
    s.desc.flags = bd.MOE_FLAG_REUSE_FWD
    rc = bd.LIB.moe_bwd(ctypes.byref(dy), *[ctypes.byref(a[n]) for n in ("x", "idx", "w", "W13", "W2")],
                        ctypes.byref(dx), ctypes.byref(dW13), ctypes.byref(dW2), ctypes.byref(dtw),
                        ctypes.byref(s), None)
    assert rc == bd.ERR["MOE_ERR_STATE"]
    dW2_bad = f.t((8, 256, 128), 2)
    s.desc.flags = 0
    rc = bd.LIB.moe_bwd(ctypes.byref(dy), *[ctypes.byref(a[n]) for n in ("x", "idx", "w", "W13", "W2")],
                        ctypes.byref(dx), ctypes.byref(dW13), ctypes.byref(dW2_bad), ctypes.byref(dtw),
                        ctypes.byref(s), None)
    assert rc == bd.ERR["MOE_ERR_DTYPE"]


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful without a CUDA device")
def test_valid_call_without_a_device_reports_cuda_error(bd):
    a, s = _fwd_args(bd)
    assert _call_fwd(bd, a, s) == bd.ERR["MOE_ERR_CUDA"]


def test_strerror_and_trace_api(bd):
    for code in bd.ERRORS:
        assert bd.strerror(code)
    assert "unknown" in bd.strerror(-1234)
    bd.moe_trace_reset()
    assert bd.moe_trace_read() == {}


def test_fp8_bwd_layout_has_only_the_backward_mxfp8_copies(bd):
    """fp8_bwd (BF16 forward, MXFP8 backward): the forward-only E4M3 copies take no scratch."""
    d = bd.make_desc(2048, 512, 256, 16, 4, bd.MOE_FP8_BWD)
    m = bd.make_desc(2048, 512, 256, 16, 4, bd.MOE_MXFP8)
    b = bd.make_desc(2048, 512, 256, 16, 4, bd.MOE_BF16)
    for name in ("x_r", "x_r_sf", "h_r", "h_r_sf", "w13_r", "w13_r_sf", "w2_r", "w2_r_sf"):
        assert bd.view_span(d, bd.MX_VIEWS[name])[1] == 0, name
        assert bd.view_span(m, bd.MX_VIEWS[name])[1] > 0, name
    for name in ("x_c", "dy_r", "dy_c", "dg_r", "dg_c", "hw_c", "w13_c", "w2_c"):
        assert bd.view_span(d, bd.MX_VIEWS[name])[1] == bd.view_span(m, bd.MX_VIEWS[name])[1] > 0, name
    assert bd.moe_scratch_bytes(b) < bd.moe_scratch_bytes(d) < bd.moe_scratch_bytes(m)


def test_fp8_fp4_layout_has_only_the_forward_copies_with_packed_weights(bd):
    """FP8 x FP4 (forward only): no backward copies; the weights' values take half the bytes of
    their E4M3 copies (two E2M1 values a byte), their scales the same bytes."""
    d = bd.make_desc(2048, 512, 256, 16, 4, bd.MOE_FP8_FP4)
    m = bd.make_desc(2048, 512, 256, 16, 4, bd.MOE_MXFP8)
    for name in ("x_c", "dy_r", "dy_c", "dg_r", "dg_c", "hw_c", "w13_c", "w2_c"):
        assert bd.view_span(d, bd.MX_VIEWS[name])[1] == 0, name
        assert bd.view_span(d, bd.MX_VIEWS[name + "_sf"])[1] == 0, name
    for name in ("x_r", "h_r"):
        assert bd.view_span(d, bd.MX_VIEWS[name])[1] == bd.view_span(m, bd.MX_VIEWS[name])[1] > 0, name
    for name in ("w13_r", "w2_r"):
        assert 2 * bd.view_span(d, bd.MX_VIEWS[name])[1] == bd.view_span(m, bd.MX_VIEWS[name])[1] > 0, name
        assert bd.view_span(d, bd.MX_VIEWS[name + "_sf"])[1] == bd.view_span(m, bd.MX_VIEWS[name + "_sf"])[1]
        off, n = bd.view_span(d, bd.MX_VIEWS[name])
        assert off % 32 == 0 and n > 0      # packed rows are read by 32-byte aligned tensor maps
    assert bd.moe_scratch_bytes(d) < bd.moe_scratch_bytes(m)


def test_fp8_fp4_backward_is_refused_before_any_launch(bd):
    f = _Fake(bd)
    T, H, I, E, k = 256, 256, 128, 8, 2
    B16, I32, F32 = bd.MOE_DT_BF16, bd.MOE_DT_I32, bd.MOE_DT_F32
    args = [f.t((T, H), B16), f.t((T, H), B16), f.t((T, k), I32), f.t((T, k), F32), f.t((E, 2 * I, H), B16),
            f.t((E, H, I), B16), f.t((T, H), B16), f.t((E, 2 * I, H), F32), f.t((E, H, I), F32), f.t((T, k), F32)]
    s = bd.MoeScratch()
    s.desc = bd.make_desc(T, H, I, E, k, bd.MOE_FP8_FP4)
    s.bytes = bd.moe_scratch_bytes(s.desc)
    s.data = 1 << 40
    assert bd.LIB.moe_bwd(*[ctypes.byref(a) for a in args], ctypes.byref(s), None) == bd.ERR["MOE_ERR_UNSUPPORTED"]
    s.desc = bd.make_desc(T, H, I, E, k, 4)     # no such precision
    assert bd.LIB.moe_bwd(*[ctypes.byref(a) for a in args], ctypes.byref(s), None) == bd.ERR["MOE_ERR_UNSUPPORTED"]


def test_router_argument_checks(bd):
    """Every bad argument of the router entry points is refused before any launch (no GPU)."""
    f = _Fake(bd)
    F32, I32, B16 = bd.MOE_DT_F32, bd.MOE_DT_I32, bd.MOE_DT_BF16
    E = bd.ERR

    def fwd(lg, idx, w):
        return bd.LIB.moe_router_fwd(ctypes.byref(lg), ctypes.byref(idx), ctypes.byref(w), None)

    def bwd(idx, w, dw, dl):
        return bd.LIB.moe_router_bwd(ctypes.byref(idx), ctypes.byref(w), ctypes.byref(dw), ctypes.byref(dl), None)
    assert fwd(f.t((64, 128), F32), f.t((64, 33), I32), f.t((64, 33), F32)) == E["MOE_ERR_UNSUPPORTED"]   # k > 32
    assert fwd(f.t((64, 4), F32), f.t((64, 8), I32), f.t((64, 8), F32)) == E["MOE_ERR_UNSUPPORTED"]       # k > E
    assert fwd(f.t((64, 2048), F32), f.t((64, 8), I32), f.t((64, 8), F32)) == E["MOE_ERR_UNSUPPORTED"]    # E > 1024
    assert fwd(f.t((64, 128), F32), f.t((32, 8), I32), f.t((64, 8), F32)) == E["MOE_ERR_SHAPE"]
    assert fwd(f.t((64, 128), F32), f.t((64, 8), I32), f.t((64, 4), F32)) == E["MOE_ERR_SHAPE"]
    assert fwd(f.t((64, 128), B16), f.t((64, 8), I32), f.t((64, 8), F32)) == E["MOE_ERR_DTYPE"]
    assert fwd(f.t((64, 128), F32), f.t((64, 8), F32), f.t((64, 8), F32)) == E["MOE_ERR_DTYPE"]
    assert fwd(f.t((64, 128), F32, contiguous=False), f.t((64, 8), I32), f.t((64, 8), F32)) == E["MOE_ERR_LAYOUT"]
    assert fwd(f.t((64, 128), F32, misalign=4), f.t((64, 8), I32), f.t((64, 8), F32)) == E["MOE_ERR_ALIGN"]
    assert bd.LIB.moe_router_fwd(None, None, None, None) == E["MOE_ERR_NULL"]
    assert bwd(f.t((64, 8), I32), f.t((64, 8), F32), f.t((64, 8), F32), f.t((64, 100), B16)) == E["MOE_ERR_DTYPE"]
    assert bwd(f.t((64, 8), I32), f.t((64, 8), F32), f.t((64, 7), F32), f.t((64, 100), F32)) == E["MOE_ERR_SHAPE"]
    assert bwd(f.t((64, 8), I32), f.t((64, 8), F32), f.t((64, 8), F32), f.t((63, 100), F32)) == E["MOE_ERR_SHAPE"]
    assert bd.LIB.moe_router_bwd(None, None, None, None, None) == E["MOE_ERR_NULL"]


def _bwd_call(bd, a, s, T=256, H=256, I=128, E=8, k=2):
    f = _Fake(bd)
    f.addr = 1 << 36
    dy = f.t((T, H), 0); dx = f.t((T, H), 0)
    dW13 = f.t((E, 2 * I, H), 1); dW2 = f.t((E, H, I), 1); dtw = f.t((T, k), 1)
    return bd.LIB.moe_bwd(ctypes.byref(dy), *[ctypes.byref(a[n]) for n in ("x", "idx", "w", "W13", "W2")],
                          ctypes.byref(dx), ctypes.byref(dW13), ctypes.byref(dW2), ctypes.byref(dtw),
                          ctypes.byref(s), None)


def test_epoch_invalidates_a_saved_forward(bd):
    """A forward saved at one epoch is not reused at another: the caller advances the epoch when
    its buffers change in place (an optimizer step), and MOE_FLAG_REUSE_FWD then refuses."""
    a, s = _fwd_args(bd, T=0)
    s.desc.flags = bd.MOE_FLAG_SAVE_GU
    assert _call_fwd(bd, a, s) == bd.ERR["MOE_OK"]                 # T = 0: records the forward, launches nothing
    s.desc.flags = bd.MOE_FLAG_REUSE_FWD
    ok = _bwd_call(bd, a, s, T=0)
    assert ok in (bd.ERR["MOE_OK"], bd.ERR["MOE_ERR_CUDA"])       # past the state check (zeroing dW needs a GPU)
    s.epoch += 1
    assert _bwd_call(bd, a, s, T=0) == bd.ERR["MOE_ERR_STATE"]
    s.epoch -= 1
    assert _bwd_call(bd, a, s, T=0) == ok


def test_weight_reuse_without_copies_is_refused_before_any_launch(bd):
    for prec in (bd.MOE_MXFP8, bd.MOE_FP8_FP4):
        a, s = _fwd_args(bd)
        s.desc.precision = prec
        s.bytes = bd.moe_scratch_bytes(s.desc)
        s.desc.flags = bd.MOE_FLAG_REUSE_WEIGHTS
        assert _call_fwd(bd, a, s) == bd.ERR["MOE_ERR_STATE"]
    a, s = _fwd_args(bd)
    s.desc.precision = bd.MOE_FP8_BWD
    s.bytes = bd.moe_scratch_bytes(s.desc)
    s.desc.flags = bd.MOE_FLAG_REUSE_WEIGHTS
    assert _bwd_call(bd, a, s) == bd.ERR["MOE_ERR_STATE"]


def test_set_wait_limit_arguments(bd):
    s = bd.MoeScratch()
    assert bd.LIB.moe_set_wait_limit(None, 0, 0) == bd.ERR["MOE_ERR_NULL"]
    assert bd.LIB.moe_set_wait_limit(ctypes.byref(s), -1, 0) == bd.ERR["MOE_ERR_SHAPE"]
    assert bd.LIB.moe_set_wait_limit(ctypes.byref(s), 12345, 0xFF) == bd.ERR["MOE_OK"]
    assert (s.state[2], s.state[3]) == (12345, bd.MOE_TEST_WITHHOLD_LOADS)   # unknown flags dropped
    assert bd.LIB.moe_set_wait_limit(ctypes.byref(s), 0, 0) == bd.ERR["MOE_OK"]
    assert (s.state[2], s.state[3]) == (0, 0)
