"""Router (the step before the layer) against the fp64 oracle: top-k of fp32 logits with the
softmax over the selected, and its backward.

Bar: expert indices bit-exact (every comparison is exact in fp32 on both sides, ties to the lower
index); weights and dlogits within 2e-6 relative (fp32 exp and a k-term fp32 sum against fp64);
the chain router -> layer -> layer backward -> router backward within the BF16 layer's 1e-2."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, f64, rel_fro, to_dev

pytestmark = pytest.mark.gpu

SHAPES = {
    "qwen3_30b": gen.custom_config("router_30b", T=16384, H=256, I=128, E=128, k=8, seed=41),
    "tiny": gen.custom_config("router_tiny", T=256, H=256, I=128, E=8, k=2, seed=42),
    "max": gen.custom_config("router_max", T=1000, H=256, I=128, E=1024, k=32, seed=43),
    "ragged_E": gen.custom_config("router_ragged", T=777, H=256, I=128, E=100, k=5, seed=44),
    "k_eq_E": gen.custom_config("router_keqe", T=64, H=256, I=128, E=32, k=32, seed=45),
}


def _run(bd, logits, k, dtw):
    T, E = logits.shape
    lg = to_dev(logits)
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    dl = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    bd.moe_router_fwd(lg, idx, w)
    bd.moe_router_bwd(idx, w, to_dev(dtw), dl)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy(), dl.cpu().numpy()


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("ties", [False, True])
def test_router_forward_and_backward(cuda_lib, name, ties):
    cfg = SHAPES[name]
    logits, dtw = gen.router_inputs(cfg, tie_step=0.25 if ties else 0.0)
    idx, w, dl = _run(cuda_lib, logits, cfg.k, dtw)
    idx_o, w_o = oracle.router_forward(logits, cfg.k)
    np.testing.assert_array_equal(idx, idx_o)
    np.testing.assert_allclose(w, w_o, rtol=2e-6, atol=1e-7)
    dl_o = oracle.router_backward(idx, w, dtw, cfg.E)       # the same fp32 weights on both sides
    np.testing.assert_allclose(dl, dl_o, rtol=2e-6, atol=2e-7)
    assert np.count_nonzero(dl) <= cfg.T * cfg.k


def test_router_empty(cuda_lib):
    _run(cuda_lib, np.zeros((0, 64), np.float32), 4, np.zeros((0, 4), np.float32))


def test_router_layer_chain(cuda_lib):
    """logits -> router -> layer forward/backward -> router backward, against the oracle chain."""
    cfg = gen.CONFIGS["tiny"]
    logits, _ = gen.router_inputs(cfg)
    inp = gen.make_inputs(cfg)
    idx_o, w_o = oracle.router_forward(logits, cfg.k)
    inp = dataclasses.replace(inp, topk_idx=idx_o, topk_w=w_o.astype(np.float32))
    L = DeviceLayer(cuda_lib, inp)
    cuda_lib.moe_router_fwd(to_dev(logits), L.idx, L.w)      # the layer consumes the GPU router's output
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD)
    dl = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device="cuda")
    cuda_lib.moe_router_bwd(L.idx, L.w, L.dtw, dl)
    torch.cuda.synchronize()
    assert L.status() == 0
    np.testing.assert_array_equal(L.idx.cpu().numpy(), idx_o)
    args = (inp.f64("x"), idx_o, w_o, inp.f64("W13"), inp.f64("W2"))
    ref = oracle.backward(inp.f64("dy"), *args)
    dl_o = oracle.router_backward(idx_o, w_o, ref["dtopk_w"], cfg.E)
    assert rel_fro(f64(dl), dl_o) < 1e-2
    assert rel_fro(f64(L.y), oracle.forward(*args)) < 1e-2
