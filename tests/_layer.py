"""Helpers shared by the GPU tests: seeded inputs to device tensors, one call of the layer
through the C ABI binding, and the comparison metrics."""
from __future__ import annotations

import numpy as np
import torch


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def rel_fro(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def max_row_rel(got, ref, floor: float = 0.1) -> float:
    """Largest relative error of any row (last axis): ||got_r - ref_r|| / max(||ref_r||, floor * rms
    row norm).  The floor keeps rows whose reference is zero (or nearly) from dividing by zero while
    still requiring their output to be near zero.  Beside the whole-tensor Frobenius error this
    catches a handful of wrong rows, which a large tensor's Frobenius norm could absorb."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    g = got.reshape(-1, got.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r, axis=1)
    rms = float(np.sqrt(np.mean(rn ** 2))) if rn.size else 0.0
    den = np.maximum(rn, max(floor * rms, 1e-300))
    return float(np.max(np.linalg.norm(g - r, axis=1) / den)) if rn.size else 0.0


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DeviceLayer:
    """Device copies of one LayerInputs plus output buffers and a scratch buffer."""

    def __init__(self, bd, inp, wgrad_dtype=torch.bfloat16):
        cfg = inp.cfg
        self.bd, self.cfg, self.inp = bd, cfg, inp
        self.x = to_dev(inp.x)
        self.idx = to_dev(inp.topk_idx)
        self.w = to_dev(inp.topk_w)
        self.W13 = to_dev(inp.W13)
        self.W2 = to_dev(inp.W2)
        self.dy = to_dev(inp.dy)
        T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
        dev = self.x.device
        self.y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        self.dx = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=dev)
        self.dW13 = torch.full((E, 2 * I, H), float("nan"), dtype=wgrad_dtype, device=dev)
        self.dW2 = torch.full((E, H, I), float("nan"), dtype=wgrad_dtype, device=dev)
        self.dtw = torch.full((T, k), float("nan"), dtype=torch.float32, device=dev)
        prec = {"bf16": bd.MOE_BF16, "mxfp8": bd.MOE_MXFP8, "fp8_bwd": bd.MOE_FP8_BWD,
                "fp8_fp4": bd.MOE_FP8_FP4}[cfg.precision]
        self.scratch = bd.Scratch(T, H, I, E, k, precision=prec, device=dev)

    def fwd(self, flags=0):
        self.bd.moe_fwd(self.x, self.idx, self.w, self.W13, self.W2, self.y, self.scratch, flags=flags)

    def bwd(self, flags=0):
        self.bd.moe_bwd(self.dy, self.x, self.idx, self.w, self.W13, self.W2, self.dx, self.dW13, self.dW2,
                        self.dtw, self.scratch, flags=flags)

    def status(self) -> int:
        return self.bd.moe_read_device_status(self.scratch)

    def view(self, which, dtype, shape):
        return self.scratch.view(which, dtype, shape)

    def rows(self):
        return (self.cfg.S + 127) // 128 * 128 + 128 * self.cfg.E


# ---- MXFP8 decoding (E4M3 code table from its bit fields; scale atoms as the header documents)
def e4m3_table() -> np.ndarray:
    tab = np.zeros(256)
    for code in range(256):
        sg, ex, m = code >> 7, (code >> 3) & 0xF, code & 7
        if ex == 0xF and m == 7:
            tab[code] = np.nan
            continue
        v = (m / 8.0) * 2.0 ** -6 if ex == 0 else (1 + m / 8.0) * 2.0 ** (ex - 7)
        tab[code] = -v if sg else v
    return tab


def sf_index(mn, kb, k_atoms):
    return ((mn // 128) * k_atoms + kb // 4) * 512 + 16 * (mn % 32) + 4 * ((mn // 32) % 4) + kb % 4


def decode_mx(q: np.ndarray, sf: np.ndarray, along: str) -> np.ndarray:
    """Dequantise an E4M3 [R, C] array with its scale atoms; along='row' (blocks of 32 columns)
    or 'col' (blocks of 32 rows)."""
    R, C = q.shape
    vals = e4m3_table()[q]
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    if along == "row":
        idx = sf_index(r, c // 32, C // 128)
    else:
        idx = sf_index(c, r // 32, R // 128)
    return vals * np.ldexp(1.0, sf[idx].astype(np.int64) - 127)


# ---- MXFP4 decoding (E2M1 code table from its bit fields: 1 sign, 2 exponent (bias 1), 1 mantissa)
def e2m1_table() -> np.ndarray:
    tab = np.zeros(16)
    for code in range(16):
        sg, ex, m = code >> 3, (code >> 1) & 3, code & 1
        v = m * 0.5 if ex == 0 else (1 + m / 2.0) * 2.0 ** (ex - 1)
        tab[code] = -v if sg else v
    return tab


def decode_mxfp4_rows(q: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Dequantise packed E2M1 [R, C/2] (the even column in the low nibble) with row-blocked scale
    atoms (blocks of 32 columns) into fp64 [R, C]."""
    R, half = q.shape
    C = 2 * half
    codes = np.empty((R, C), dtype=np.int64)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    r = np.arange(R)[:, None]
    c = np.arange(C)[None, :]
    return e2m1_table()[codes] * np.ldexp(1.0, sf[sf_index(r, c // 32, C // 128)].astype(np.int64) - 127)
