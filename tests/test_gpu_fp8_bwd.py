"""fp8_bwd precision (the pages' BF16 forward with an FP8 backward, FP8 read as MXFP8 on
Blackwell) against the fp64 oracle in the same mode.

Bar: the forward is bit-identical to the BF16 layer's (the same kernels run); dx, dW13, dW2 and
dtopk_w within a relative Frobenius error of 3e-2 of the oracle that quantises the backward
GEMMs' operands as the MXFP8 backward does and keeps the forward exact."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, f64, rel_fro

pytestmark = pytest.mark.gpu
TOL = 3e-2


def fp8b(cfg):
    return dataclasses.replace(cfg, precision="fp8_bwd", name=cfg.name + "_fp8b")


SMALL = {
    "tiny": fp8b(gen.CONFIGS["tiny"]),
    "medium": fp8b(gen.custom_config("medium", T=2048, H=512, I=256, E=16, k=4, seed=21)),
    "medium_I384": fp8b(gen.custom_config("medium_I384", T=1500, H=768, I=384, E=12, k=3, seed=22)),
    "skew_small": fp8b(gen.custom_config("skew_small", T=1024, H=256, I=128, E=32, k=8, routing="zipf", seed=23)),
}


def _args(inp):
    return inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2")


@pytest.mark.parametrize("name", ["tiny", "medium"])
def test_forward_is_the_bf16_forward(cuda_lib, name):
    inp = gen.make_inputs(SMALL[name])
    A = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    B = DeviceLayer(cuda_lib, gen.make_inputs(dataclasses.replace(SMALL[name], precision="bf16")))
    A.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    B.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    torch.cuda.synchronize()
    assert A.status() == 0 and B.status() == 0
    assert torch.equal(A.y, B.y)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("reuse", [False, True])
def test_backward(cuda_lib, name, reuse):
    inp = gen.make_inputs(SMALL[name])
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    flags = 0
    if reuse:
        L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
        flags = cuda_lib.MOE_FLAG_REUSE_FWD
    L.bwd(flags=flags)
    torch.cuda.synchronize()
    assert L.status() == 0
    ref = oracle.backward(inp.f64("dy"), *_args(inp), fp8_bwd=True)
    bf = oracle.backward(inp.f64("dy"), *_args(inp))
    for got, n in ((L.dx, "dx"), (L.dW13, "dW13"), (L.dW2, "dW2"), (L.dtw, "dtopk_w")):
        err = rel_fro(f64(got), ref[n])
        assert err < TOL, (n, err)
    # and the backward is an MXFP8 one: closer to the quantised oracle than to the BF16 one
    assert rel_fro(f64(L.dx), ref["dx"]) < rel_fro(f64(L.dx), bf["dx"])


@pytest.mark.parametrize("name", ["qwen3_30b_a3b", "qwen3_235b_a22b"])
def test_full_size_sampled(cuda_lib, name):
    cfg = fp8b(gen.CONFIGS[name])
    inp = gen.make_inputs(cfg)
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.fwd()
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD)
    torch.cuda.synchronize()
    assert L.status() == 0
    rng = np.random.default_rng(2)
    toks = np.sort(rng.choice(cfg.T, 8, replace=False))
    x, dy, W13, W2 = inp.f32("x"), inp.f32("dy"), inp.f32("W13"), inp.f32("W2")
    ti = torch.from_numpy(toks).cuda()
    y_s = oracle.forward_tokens(x, inp.topk_idx, inp.topk_w, W13, W2, toks)
    assert rel_fro(f64(L.y[ti]), y_s) < 1e-2
    dx_s, dtw_s = oracle.backward_tokens(dy, x, inp.topk_idx, inp.topk_w, W13, W2, toks, fp8_bwd=True)
    assert rel_fro(f64(L.dx[ti]), dx_s) < TOL
    assert rel_fro(f64(L.dtw[ti]), dtw_s) < TOL
    experts = [0, int(rng.integers(cfg.E))]
    for e, (a13, a2) in zip(experts, oracle.wgrad_experts(dy, x, inp.topk_idx, inp.topk_w, W13, W2, experts,
                                                          fp8_bwd=True)):
        assert rel_fro(f64(L.dW13[e]), a13) < TOL, e
        assert rel_fro(f64(L.dW2[e]), a2) < TOL, e
    for t in (L.y, L.dx, L.dW13, L.dW2, L.dtw):
        assert torch.isfinite(t).all()
