"""Parity of the CUDA path (called through the C ABI) with the fp64 oracle.

Bar: routing outputs (counts, offsets, reorder and inverse) bit-exact; y, dx, dW13, dW2 and dtopk_w
within a relative Frobenius error of 1e-2 (BF16), on the same seeded inputs.  Small configurations
are compared element by element in full, and there every row of y, dx, dW13, dW2 must also be
within ROW_TOL: each output and each bf16 intermediate rounds once to 8 significant bits (about
2^-8 / sqrt(3) relative in rms), so a row of at least 128 elements lands well inside 2e-2, while a
wrong row is off by order one.  The full-size workloads are compared on sampled tokens and experts
the oracle evaluates one by one."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, f64, max_row_rel, rel_fro

pytestmark = pytest.mark.gpu
TOL = 1e-2
ROW_TOL = 2e-2

SMALL = {
    "tiny": gen.CONFIGS["tiny"],
    # several m- and n-tiles per expert with ragged tails, K over several pipeline rounds
    "medium": gen.custom_config("medium", T=2048, H=512, I=256, E=16, k=4, seed=21),
    "medium_I384": gen.custom_config("medium_I384", T=1500, H=768, I=384, E=12, k=3, seed=22),
    # wide I: four n-tiles of the forward gate/up and two of the backward down per m-tile
    "medium_I512": gen.custom_config("medium_I512", T=1024, H=256, I=512, E=8, k=2, seed=24),
    "skew_small": gen.custom_config("skew_small", T=1024, H=256, I=128, E=32, k=8, routing="zipf", seed=23),
    # k > 32: the token-major gather loads a token's destinations 32 at a time
    "wide_k": gen.custom_config("wide_k", T=96, H=256, I=128, E=48, k=36, seed=25),
}


def _oracle_args(inp):
    return inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2")


def _check_routing(L, inp):
    cfg = inp.cfg
    r = oracle.route(inp.topk_idx, cfg.E)
    E, S = cfg.E, cfg.S
    bd = L.bd
    cnt = L.view(bd.MOE_VIEW_COUNTS, torch.int32, (E,)).cpu().numpy()
    off = L.view(bd.MOE_VIEW_OFFSETS, torch.int32, (E + 1,)).cpu().numpy()
    perm = L.view(bd.MOE_VIEW_PERM, torch.int32, (S,)).cpu().numpy()
    inv = L.view(bd.MOE_VIEW_INV, torch.int32, (S,)).cpu().numpy()
    pad = L.view(bd.MOE_VIEW_PAD_OFFSETS, torch.int32, (E + 1,)).cpu().numpy()
    np.testing.assert_array_equal(cnt, r["cnt"])
    np.testing.assert_array_equal(off, r["off"])
    np.testing.assert_array_equal(perm, r["perm"])
    np.testing.assert_array_equal(inv, r["inv"])
    np.testing.assert_array_equal(pad, np.concatenate([[0], np.cumsum(-(-r["cnt"] // 128) * 128)]))
    return r, pad


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_and_intermediates(cuda_lib, name):
    inp = gen.make_inputs(SMALL[name])
    cfg = inp.cfg
    L = DeviceLayer(cuda_lib, inp)
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    torch.cuda.synchronize()
    assert L.status() == 0
    r, pad = _check_routing(L, inp)
    y_ref, fw = oracle.forward(*_oracle_args(inp), keep=True)
    assert rel_fro(f64(L.y), y_ref) < TOL
    assert max_row_rel(f64(L.y), y_ref) < ROW_TOL
    # padded-layout intermediates: row of sorted position p of expert e sits at pad[e] + (p - off[e])
    R = L.rows()
    prow = np.empty(cfg.S, dtype=np.int64)
    for e in range(cfg.E):
        lo, hi = r["off"][e], r["off"][e + 1]
        prow[lo:hi] = pad[e] + np.arange(hi - lo)
    xperm = L.view(cuda_lib.MOE_VIEW_XPERM, torch.bfloat16, (R, cfg.H))
    np.testing.assert_array_equal(f64(xperm[torch.from_numpy(prow).cuda()]), fw["X_perm"])
    padmask = np.ones(int(pad[-1]), dtype=bool)
    padmask[prow] = False
    assert torch.all(xperm[:int(pad[-1])][torch.from_numpy(padmask).cuda()] == 0)
    gu = f64(L.view(cuda_lib.MOE_VIEW_GU, torch.bfloat16, (R, 2 * cfg.I))[torch.from_numpy(prow).cuda()])
    assert rel_fro(gu[:, :cfg.I], fw["g"]) < TOL and rel_fro(gu[:, cfg.I:], fw["u"]) < TOL
    # the gate/up epilogue stores w h (the routing weight applied before the down product)
    hid = f64(L.view(cuda_lib.MOE_VIEW_HID, torch.bfloat16, (R, cfg.I))[torch.from_numpy(prow).cuda()])
    assert rel_fro(hid, fw["w_sorted"][:, None] * fw["h"]) < TOL
    ypart = f64(L.view(cuda_lib.MOE_VIEW_YPART, torch.bfloat16, (R, cfg.H))[torch.from_numpy(prow).cuda()])
    assert rel_fro(ypart, fw["w_sorted"][:, None] * fw["o"]) < TOL


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("reuse", [False, True])
def test_backward(cuda_lib, name, reuse):
    inp = gen.make_inputs(SMALL[name])
    L = DeviceLayer(cuda_lib, inp)
    if reuse:
        L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD if reuse else 0)
    torch.cuda.synchronize()
    assert L.status() == 0
    ref = oracle.backward(inp.f64("dy"), *_oracle_args(inp))
    for got, name_ in ((L.dx, "dx"), (L.dW13, "dW13"), (L.dW2, "dW2"), (L.dtw, "dtopk_w")):
        err = rel_fro(f64(got), ref[name_])
        assert err < TOL, (name_, err)
        if name_ != "dtopk_w":                 # rows of k values: a per-row norm means little
            row = max_row_rel(f64(got), ref[name_])
            assert row < ROW_TOL, (name_, row)


def test_backward_intermediates(cuda_lib):
    inp = gen.make_inputs(SMALL["medium"])
    cfg = inp.cfg
    L = DeviceLayer(cuda_lib, inp)
    L.bwd()
    torch.cuda.synchronize()
    r, pad = _check_routing(L, inp)
    ref = oracle.backward(inp.f64("dy"), *_oracle_args(inp), keep=True)
    prow = np.empty(cfg.S, dtype=np.int64)
    for e in range(cfg.E):
        lo, hi = r["off"][e], r["off"][e + 1]
        prow[lo:hi] = pad[e] + np.arange(hi - lo)
    idx = torch.from_numpy(prow).cuda()
    R = L.rows()
    dG = f64(L.view(cuda_lib.MOE_VIEW_DG, torch.bfloat16, (R, 2 * cfg.I))[idx])
    hw = f64(L.view(cuda_lib.MOE_VIEW_HW, torch.bfloat16, (R, cfg.I))[idx])
    dyp = f64(L.view(cuda_lib.MOE_VIEW_DYPERM, torch.bfloat16, (R, cfg.H))[idx])
    np.testing.assert_array_equal(dyp, ref["dY_perm"])
    assert rel_fro(dG, ref["dG"]) < TOL
    assert rel_fro(hw, ref["Hw"]) < TOL


def test_reuse_matches_recompute_bitwise(cuda_lib):
    inp = gen.make_inputs(SMALL["medium"])
    A = DeviceLayer(cuda_lib, inp)
    A.bwd()
    B = DeviceLayer(cuda_lib, inp)
    B.fwd()                                   # a forward without the save, then one with it
    B.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    B.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD)
    torch.cuda.synchronize()
    for a, b in ((A.dx, B.dx), (A.dW13, B.dW13), (A.dW2, B.dW2), (A.dtw, B.dtw)):
        assert torch.equal(a, b)


def test_reuse_refused_after_other_inputs(cuda_lib):
    inp = gen.make_inputs(SMALL["tiny"])
    L = DeviceLayer(cuda_lib, inp)
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.x = L.x.clone()
    with pytest.raises(cuda_lib.MoeError) as ei:
        L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD)
    assert ei.value.code == cuda_lib.ERR["MOE_ERR_STATE"]


def test_deterministic(cuda_lib):
    inp = gen.make_inputs(SMALL["skew_small"])
    L = DeviceLayer(cuda_lib, inp)
    L.fwd(); L.bwd()
    torch.cuda.synchronize()
    first = [t.clone() for t in (L.y, L.dx, L.dW13, L.dW2, L.dtw)]
    L.fwd(); L.bwd()
    torch.cuda.synchronize()
    for a, b in zip(first, (L.y, L.dx, L.dW13, L.dW2, L.dtw)):
        assert torch.equal(a, b)


def test_fp32_weight_grads(cuda_lib):
    inp = gen.make_inputs(SMALL["medium"])
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.bwd()
    torch.cuda.synchronize()
    ref = oracle.backward(inp.f64("dy"), *_oracle_args(inp))
    assert rel_fro(f64(L.dW13), ref["dW13"]) < TOL
    assert rel_fro(f64(L.dW2), ref["dW2"]) < TOL


# ---------------------------------------------------------------- edge cases
def _routed(cfg, idx):
    inp = gen.make_inputs(cfg)
    inp.topk_idx = np.ascontiguousarray(idx.astype(np.int32))
    return inp


@pytest.mark.parametrize("case", ["one_token", "all_on_one_expert", "empty_experts", "single_expert_top1",
                                  "fewer_rows_than_a_tile", "max_experts"])
def test_edge_cases(cuda_lib, case):
    if case == "one_token":
        inp = gen.make_inputs(gen.custom_config(T=1, H=256, I=128, E=8, k=2, seed=31))
    elif case == "all_on_one_expert":
        cfg = gen.custom_config(T=300, H=256, I=128, E=8, k=1, seed=32)
        inp = _routed(cfg, np.full((300, 1), 5))
    elif case == "empty_experts":
        cfg = gen.custom_config(T=400, H=256, I=256, E=16, k=2, seed=33)
        idx = np.stack([np.arange(400) % 3, 7 + np.arange(400) % 2], axis=1)     # 11 experts idle
        inp = _routed(cfg, idx)
    elif case == "single_expert_top1":
        inp = gen.make_inputs(gen.custom_config(T=200, H=256, I=128, E=1, k=1, seed=34))
    elif case == "max_experts":
        # the largest expert count the layer takes (1024): about four rows per expert, some idle
        inp = gen.make_inputs(gen.custom_config(T=512, H=256, I=128, E=1024, k=8, seed=38))
    else:
        inp = gen.make_inputs(gen.custom_config(T=20, H=512, I=256, E=4, k=2, seed=35))
    L = DeviceLayer(cuda_lib, inp)
    L.fwd()
    L.bwd()
    torch.cuda.synchronize()
    assert L.status() == 0
    _check_routing(L, inp)
    y = oracle.forward(*_oracle_args(inp))
    ref = oracle.backward(inp.f64("dy"), *_oracle_args(inp))
    assert rel_fro(f64(L.y), y) < TOL
    for got, n in ((L.dx, "dx"), (L.dW13, "dW13"), (L.dW2, "dW2"), (L.dtw, "dtopk_w")):
        if np.linalg.norm(ref[n]) == 0:
            assert torch.all(got == 0), n
        else:
            assert rel_fro(f64(got), ref[n]) < TOL, n
    if case in ("empty_experts", "max_experts"):
        idle = sorted(set(range(inp.cfg.E)) - set(np.unique(inp.topk_idx).tolist()))
        assert torch.all(L.dW13[idle] == 0) and torch.all(L.dW2[idle] == 0)


def test_zero_tokens(cuda_lib):
    inp = gen.make_inputs(gen.custom_config(T=0, H=256, I=128, E=8, k=2, seed=36))
    L = DeviceLayer(cuda_lib, inp)
    L.fwd()
    L.bwd()
    torch.cuda.synchronize()
    assert torch.all(L.dW13 == 0) and torch.all(L.dW2 == 0)


def test_bad_expert_ids_are_flagged_not_used(cuda_lib):
    cfg = gen.custom_config(T=256, H=256, I=128, E=8, k=2, seed=37)
    inp = gen.make_inputs(cfg)
    idx = inp.topk_idx.copy()
    idx[3, 0] = 8
    idx[10, 1] = -1
    inp.topk_idx = idx
    L = DeviceLayer(cuda_lib, inp)
    L.fwd()
    torch.cuda.synchronize()
    assert L.status() == cuda_lib.MOE_DEV_BAD_EXPERT
    assert L.status() == 0                     # reading clears the word
    # dropped slots: inv = -1, and the two positions they free at the end of perm hold -1
    S = cfg.S
    inv = L.view(cuda_lib.MOE_VIEW_INV, torch.int32, (S,)).cpu().numpy()
    perm = L.view(cuda_lib.MOE_VIEW_PERM, torch.int32, (S,)).cpu().numpy()
    assert inv[3 * 2 + 0] == -1 and inv[10 * 2 + 1] == -1
    assert np.array_equal(perm[S - 2:], [-1, -1]) and (perm[:S - 2] >= 0).all()
    assert np.array_equal(inv[perm[:S - 2]], np.arange(S - 2))
    # the valid slots still produce the layer over the valid slots only
    keep = (idx >= 0) & (idx < 8)
    w = np.where(keep, inp.topk_w, 0.0)
    y_ref = oracle.forward(inp.f64("x"), np.where(keep, idx, 0), w, inp.f64("W13"), inp.f64("W2"))
    assert rel_fro(f64(L.y), y_ref) < TOL


# ---------------------------------------------------------------- full-size workloads, sampled
FULL = ["qwen3_30b_a3b", "skew_zipf_16k", "skew_zipf_4k", "qwen3_235b_a22b"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(cuda_lib, name):
    cfg = gen.CONFIGS[name]
    inp = gen.make_inputs(cfg)
    L = DeviceLayer(cuda_lib, inp)
    L.fwd()
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD)
    torch.cuda.synchronize()
    assert L.status() == 0
    r, _ = _check_routing(L, inp)
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(cfg.T, 12, replace=False))
    args = (inp.x, inp.topk_idx, inp.topk_w.astype(np.float64), inp.W13, inp.W2)
    x16, W13_16, W2_16 = inp.f32("x"), inp.W13, inp.W2
    from moe_expert_layer_permute_gb300.inputs import bf16_bits_to_f32
    Wa = bf16_bits_to_f32(inp.W13)
    Wb = bf16_bits_to_f32(inp.W2)
    dy = inp.f32("dy")
    y_s = oracle.forward_tokens(x16, inp.topk_idx, inp.topk_w, Wa, Wb, toks)
    assert rel_fro(f64(L.y[torch.from_numpy(toks).cuda()]), y_s) < TOL
    dx_s, dtw_s = oracle.backward_tokens(dy, x16, inp.topk_idx, inp.topk_w, Wa, Wb, toks)
    assert rel_fro(f64(L.dx[torch.from_numpy(toks).cuda()]), dx_s) < TOL
    assert rel_fro(f64(L.dtw[torch.from_numpy(toks).cuda()]), dtw_s) < TOL
    cnt = r["cnt"]
    experts = [int(np.argmax(cnt)), int(np.argmin(np.where(cnt > 0, cnt, 1 << 30))), int(rng.integers(cfg.E))]
    for e, (a13, a2) in zip(experts, oracle.wgrad_experts(dy, x16, inp.topk_idx, inp.topk_w, Wa, Wb, experts)):
        assert rel_fro(f64(L.dW13[e]), a13) < TOL, e
        assert rel_fro(f64(L.dW2[e]), a2) < TOL, e
    for e in np.nonzero(cnt == 0)[0]:
        assert torch.all(L.dW13[int(e)] == 0) and torch.all(L.dW2[int(e)] == 0)
    # properties that hold at any size: finite outputs everywhere
    for t in (L.y, L.dx, L.dW13, L.dW2, L.dtw):
        assert torch.isfinite(t).all()
