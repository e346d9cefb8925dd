"""The device weight quantisers (MXFP8 E4M3 and MXFP4 E2M1 copies of W13 and W2) on hand-built
blocks, against the oracle's quantise-dequantise.

Every block is scaled by 2^s for s across the E8M0 range and holds, besides one element that
fixes its scale: each midpoint between consecutive codes of the format (ties go to the even code),
the bf16 values just below and above each midpoint, values past the largest code (saturation),
E4M3 subnormals, zeros and both signs; some blocks are all zero.  x is zero, so the layer's
outputs stay finite whatever the weights, and y must be exactly zero.

Bar: the codes decode exactly to the oracle's values."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, decode_mx, decode_mxfp4_rows, e2m1_table, e4m3_table

pytestmark = pytest.mark.gpu


def _grid(fmt):
    """Non-negative finite values of the format, from its bit fields (not from the oracle)."""
    tab = e2m1_table() if fmt == "e2m1" else e4m3_table()
    v = np.unique(np.abs(tab[np.isfinite(tab)]))
    return v, float(v.max())


def _bf16_neighbours(v):
    """The bf16 values one step below and above the bf16 value v (v > 0)."""
    b = gen.f32_to_bf16_bits(np.array([v], dtype=np.float32)).astype(np.int32)
    lo = gen.bf16_bits_to_f32((b - 1).astype(np.uint16))[0]
    hi = gen.bf16_bits_to_f32((b + 1).astype(np.uint16))[0]
    return float(lo), float(hi)


def _special_values(fmt):
    grid, top = _grid(fmt)
    mids = (grid[1:] + grid[:-1]) / 2
    vals = list(grid) + list(mids)
    for m in mids:
        vals += list(_bf16_neighbours(m))
    vals += [top * 1.0625, top * 1.25, top * 1.875]   # past the largest code (same block exponent)
    return np.array(vals), top


def _blocks(n_blocks, fmt, rng):
    """n_blocks rows of 32 bf16-exact values, as described in the module docstring."""
    vals, top = _special_values(fmt)
    # lowest scales: the E4M3 subnormal midpoints and their bf16 neighbours must stay bf16-exact
    exps = [-100, -64, -9, -1, 0, 1, 5, 40, 110] if fmt == "e4m3" else [-120, -64, -3, 0, 2, 17, 90, 120]
    out = np.zeros((n_blocks, 32))
    for b in range(n_blocks):
        kind = b % 7
        if kind == 6:
            continue                                   # an all-zero block
        s = exps[(b // 7) % len(exps)]
        blk = rng.choice(vals, 32) * rng.choice([-1.0, 1.0], 32)
        blk[rng.integers(32)] = top * rng.choice([-1.0, 1.0])       # fixes the block exponent at s
        if kind == 5:
            blk[rng.integers(32)] = top * 1.875            # a saturating element that keeps it
        if kind == 4:
            blk[rng.integers(32, size=4)] = 0.0
        out[b] = np.ldexp(blk, s)
    bits = gen.f32_to_bf16_bits(out.astype(np.float32))
    assert np.array_equal(gen.bf16_bits_to_f32(bits).astype(np.float64), out), "block values must be bf16-exact"
    return bits


@pytest.mark.parametrize("precision", ["fp8_fp4", "mxfp8"])
def test_weight_quantiser_on_hand_built_blocks(cuda_lib, precision):
    bd = cuda_lib
    fmt = "e2m1" if precision == "fp8_fp4" else "e4m3"
    T, H, I, E, k = 64, 256, 128, 2, 1
    cfg = dataclasses.replace(gen.custom_config("quant_edges", T=T, H=H, I=I, E=E, k=k, seed=41), precision=precision)
    inp = gen.make_inputs(cfg)
    rng = np.random.default_rng(7)
    inp.W13 = _blocks(E * 2 * I * H // 32, fmt, rng).reshape(E, 2 * I, H)
    inp.W2 = _blocks(E * H * I // 32, fmt, rng).reshape(E, H, I)
    inp.x = np.zeros((T, H), dtype=np.uint16)
    L = DeviceLayer(bd, inp, wgrad_dtype=torch.float32)
    L.fwd()
    torch.cuda.synchronize()
    assert L.status() == 0
    assert torch.all(L.y == 0)
    W13, W2 = inp.f64("W13"), inp.f64("W2")
    sf = lambda n: L.view(bd.MX_VIEWS[n], torch.uint8, (-1,)).cpu().numpy()   # noqa: E731
    if fmt == "e2m1":
        q13 = L.view(bd.MX_VIEWS["w13_r"], torch.uint8, (E * 2 * I, H // 2)).cpu().numpy()
        d13 = decode_mxfp4_rows(q13, sf("w13_r_sf"))
        q2 = L.view(bd.MX_VIEWS["w2_r"], torch.uint8, (E * H, I // 2)).cpu().numpy()
        d2 = decode_mxfp4_rows(q2, sf("w2_r_sf"))
    else:
        q13 = L.view(bd.MX_VIEWS["w13_r"], torch.uint8, (E * 2 * I, H)).cpu().numpy()
        d13 = decode_mx(q13, sf("w13_r_sf"), "row")
        q2 = L.view(bd.MX_VIEWS["w2_r"], torch.uint8, (E * H, I)).cpu().numpy()
        d2 = decode_mx(q2, sf("w2_r_sf"), "row")
    d13 = d13.reshape(E, 2 * I // 128, 2, 64, H)           # 128-row blocks of [64 gate | 64 up]
    ref13 = oracle.mx_qdq(W13, axis=2, fmt=fmt)
    np.testing.assert_array_equal(d13[:, :, 0].reshape(E, I, H), ref13[:, :I])
    np.testing.assert_array_equal(d13[:, :, 1].reshape(E, I, H), ref13[:, I:])
    np.testing.assert_array_equal(d2.reshape(E, H, I), oracle.mx_qdq(W2, axis=2, fmt=fmt))
    if fmt == "e4m3":
        # the column-blocked copies of the MXFP8 backward too (blocks of 32 along 2I and along H)
        q13c = L.view(bd.MX_VIEWS["w13_c"], torch.uint8, (E * 2 * I, H)).cpu().numpy()
        np.testing.assert_array_equal(decode_mx(q13c, sf("w13_c_sf"), "col").reshape(E, 2 * I, H),
                                      oracle.mx_qdq(W13, axis=1))
        q2c = L.view(bd.MX_VIEWS["w2_c"], torch.uint8, (E * H, I)).cpu().numpy()
        np.testing.assert_array_equal(decode_mx(q2c, sf("w2_c_sf"), "col").reshape(E, H, I),
                                      oracle.mx_qdq(W2, axis=1))
