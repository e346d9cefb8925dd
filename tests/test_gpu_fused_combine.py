"""The combine fused into the down projection (MOE_FLAG_FUSED_COMBINE): one forward whose down
GEMM epilogue adds w * o of every routed row into an fp32 accumulator by token, with no Ypart rows
and no separate combine (the pages' single fused call: MarkTechPost, "Prime Intellect Releases
Prime Mega MoE", section "How does the fused kernel work?").

Against the fp64 oracle it must meet the same bound as the fixed-order combine, and be at least
as close (it skips the bf16 rounding of each Ypart row).  Its fp32 additions follow the tiles'
timing, so two runs may differ, but only in the rounding of y: by at most one bf16 step."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, f64, max_row_rel, rel_fro

pytestmark = pytest.mark.gpu
TOL, ROW_TOL = 1e-2, 2e-2

CASES = {
    "tiny": gen.CONFIGS["tiny"],
    "medium": gen.custom_config("medium", T=2048, H=512, I=256, E=16, k=4, seed=21),
    "k1": gen.custom_config("k1", T=1000, H=256, I=128, E=4, k=1, seed=51),
    "skew_small": gen.custom_config("skew_small", T=1024, H=256, I=128, E=32, k=8, routing="zipf", seed=23),
}


def _args(inp):
    return inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2")


@pytest.mark.parametrize("name", list(CASES))
def test_fused_combine_matches_the_oracle(cuda_lib, name):
    bd = cuda_lib
    inp = gen.make_inputs(CASES[name])
    L = DeviceLayer(bd, inp)
    L.fwd()
    y_plain = L.y.clone()
    L.fwd(flags=bd.MOE_FLAG_FUSED_COMBINE)
    torch.cuda.synchronize()
    assert L.status() == 0
    y_ref = oracle.forward(*_args(inp))
    err, err_plain = rel_fro(f64(L.y), y_ref), rel_fro(f64(y_plain), y_ref)
    assert err < TOL and max_row_rel(f64(L.y), y_ref) < ROW_TOL, err
    assert err <= err_plain * 1.05, (err, err_plain)
    # a second run: equal up to the final bf16 rounding of each element
    y1 = L.y.clone()
    L.fwd(flags=bd.MOE_FLAG_FUSED_COMBINE)
    torch.cuda.synchronize()
    a, b = f64(y1), f64(L.y)
    # one bf16 step at the element's magnitude, or a part in 1e6 of the typical |y| where the sum
    # cancels to near zero
    step = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7 + 1e-6 * np.sqrt(np.mean(a * a))
    assert (np.abs(a - b) <= step).all()


def test_fused_forward_then_backward(cuda_lib):
    """A fused saving forward leaves the same [g|u] and routing for the backward."""
    bd = cuda_lib
    inp = gen.make_inputs(CASES["medium"])
    L = DeviceLayer(bd, inp)
    L.fwd(flags=bd.MOE_FLAG_SAVE_GU | bd.MOE_FLAG_FUSED_COMBINE)
    L.bwd(flags=bd.MOE_FLAG_REUSE_FWD)
    torch.cuda.synchronize()
    assert L.status() == 0
    g = oracle.backward(inp.f64("dy"), *_args(inp))
    for name, got in (("dx", L.dx), ("dW13", L.dW13), ("dW2", L.dW2), ("dtopk_w", L.dtw)):
        assert rel_fro(f64(got), g[name]) < TOL, name


def test_fused_combine_is_bf16_forward_only(cuda_lib):
    bd = cuda_lib
    import dataclasses
    inp = gen.make_inputs(dataclasses.replace(CASES["tiny"], precision="mxfp8"))
    L = DeviceLayer(bd, inp, wgrad_dtype=torch.float32)
    with pytest.raises(bd.MoeError) as e:
        L.fwd(flags=bd.MOE_FLAG_FUSED_COMBINE)
    assert e.value.code == bd.ERR["MOE_ERR_UNSUPPORTED"]
