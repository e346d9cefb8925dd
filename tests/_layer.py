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
        self.scratch = bd.Scratch(T, H, I, E, k, device=dev)

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
        return self.cfg.S + 128 * self.cfg.E
