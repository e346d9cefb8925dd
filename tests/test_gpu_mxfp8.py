"""MXFP8 path (E4M3 values, one E8M0 scale per 32 elements along each GEMM's contraction axis)
against the fp64 oracle that applies the same quantise-dequantise rounding.

Bar: the quantiser's outputs decode exactly to the oracle's quantise-dequantise of the same
bf16 inputs; y, dx, dW13, dW2 and dtopk_w within a relative Frobenius error of 3e-2."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, decode_mx, f64, max_row_rel, rel_fro

pytestmark = pytest.mark.gpu
TOL = 3e-2
# per row of y, dx, dW13, dW2: twice the whole-tensor bound.  Against the quantise-aware oracle the
# differences (fp32 against fp64 arithmetic, a rare code flipped at a near-tie) spread over rows of
# at least 128 elements, while a wrong row is off by order one.
ROW_TOL = 6e-2


def mx(cfg):
    import dataclasses
    return dataclasses.replace(cfg, precision="mxfp8", name=cfg.name + "_mx")


SMALL = {
    "tiny": mx(gen.CONFIGS["tiny"]),
    "medium": mx(gen.custom_config("medium", T=2048, H=512, I=256, E=16, k=4, seed=21)),
    "medium_I384": mx(gen.custom_config("medium_I384", T=1500, H=768, I=384, E=12, k=3, seed=22)),
    "skew_small": mx(gen.custom_config("skew_small", T=1024, H=256, I=128, E=32, k=8, routing="zipf", seed=23)),
    # k > 32: the token-major row quantiser stores to a token's destinations 32 at a time
    "wide_k": mx(gen.custom_config("wide_k", T=96, H=256, I=128, E=48, k=36, seed=25)),
}


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_activation_quantiser_on_hand_built_blocks(cuda_lib, precision):
    """x and dy made of the weight-quantiser edge blocks (each 32-column row block holds the E4M3
    midpoints, their bf16 neighbours, saturating values, subnormals and zeros, at scales across
    the E8M0 range) with zero weights: the dispatched row-blocked and token-blocked copies decode
    exactly to the oracle's quantise-dequantise, and the padding rows hold zero codes."""
    import dataclasses

    from test_gpu_quant_edges import _blocks
    T, H, I, E, k = 192, 512, 128, 6, 2
    cfg = dataclasses.replace(gen.custom_config("act_edges", T=T, H=H, I=I, E=E, k=k, seed=43), precision=precision)
    inp = gen.make_inputs(cfg)
    rng = np.random.default_rng(11)
    inp.x = _blocks(T * H // 32, "e4m3", rng).reshape(T, H)
    inp.dy = _blocks(T * H // 32, "e4m3", rng).reshape(T, H)
    inp.W13 = np.zeros_like(inp.W13)
    inp.W2 = np.zeros_like(inp.W2)
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.bwd()
    torch.cuda.synchronize()
    assert L.status() == 0
    R = L.rows()
    r, prow = _padded_rows(L, inp)
    used = int(L.view(L.bd.MOE_VIEW_PAD_OFFSETS, torch.int32, (E + 1,)).cpu().numpy()[E])
    pad = np.setdiff1d(np.arange(used), prow)
    assert pad.size > 0
    X = inp.f64("x")[r["perm"] // k]
    dY = inp.f64("dy")[r["perm"] // k]
    views = [("x_c", X, "col"), ("dy_r", dY, "row"), ("dy_c", dY, "col")]
    if precision == "mxfp8":
        views.append(("x_r", X, "row"))
    for name, ref, kind in views:
        q, sf = _mxview(L, name, (R, H))
        expect = oracle.mx_qdq(ref, axis=1) if kind == "row" else oracle.mx_qdq_segments(ref, r["off"])
        np.testing.assert_array_equal(decode_mx(q, sf, kind)[prow], expect, err_msg=name)
        assert not q[pad].any(), name


def _args(inp):
    return inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2")


def _padded_rows(L, inp):
    bd = L.bd
    cfg = inp.cfg
    r = oracle.route(inp.topk_idx, cfg.E)
    pad = L.view(bd.MOE_VIEW_PAD_OFFSETS, torch.int32, (cfg.E + 1,)).cpu().numpy()
    prow = np.empty(cfg.S, dtype=np.int64)
    for e in range(cfg.E):
        lo, hi = r["off"][e], r["off"][e + 1]
        prow[lo:hi] = pad[e] + np.arange(hi - lo)
    return r, prow


def _mxview(L, name, shape):
    bd = L.bd
    q = L.view(bd.MX_VIEWS[name], torch.uint8, shape).cpu().numpy()
    sf = L.view(bd.MX_VIEWS[name + "_sf"], torch.uint8, (-1,)).cpu().numpy()
    return q, sf


@pytest.mark.parametrize("name", ["medium", "medium_I384", "skew_small"])
def test_quantiser_matches_oracle_bit_exact(cuda_lib, name):
    inp = gen.make_inputs(SMALL[name])
    cfg = inp.cfg
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.bwd()
    torch.cuda.synchronize()
    assert L.status() == 0
    H, I, E, R = cfg.H, cfg.I, cfg.E, L.rows()
    r, prow = _padded_rows(L, inp)
    X = inp.f64("x")[r["perm"] // cfg.k]
    dY = inp.f64("dy")[r["perm"] // cfg.k]
    # activations: along the row (K-major use) and along the tokens of each expert group
    q, sf = _mxview(L, "x_r", (R, H))
    np.testing.assert_array_equal(decode_mx(q, sf, "row")[prow], oracle.mx_qdq(X, axis=1))
    q, sf = _mxview(L, "x_c", (R, H))
    np.testing.assert_array_equal(decode_mx(q, sf, "col")[prow], oracle.mx_qdq_segments(X, r["off"]))
    q, sf = _mxview(L, "dy_c", (R, H))
    np.testing.assert_array_equal(decode_mx(q, sf, "col")[prow], oracle.mx_qdq_segments(dY, r["off"]))
    q, sf = _mxview(L, "dy_r", (R, H))
    np.testing.assert_array_equal(decode_mx(q, sf, "row")[prow], oracle.mx_qdq(dY, axis=1))
    # weights: W2 along H per expert (column blocks of [E*H, I]); W13 along H in gate/up row blocks
    W2 = inp.f64("W2")
    q, sf = _mxview(L, "w2_c", (E * H, I))
    np.testing.assert_array_equal(decode_mx(q, sf, "col").reshape(E, H, I), oracle.mx_qdq(W2, axis=1))
    q, sf = _mxview(L, "w2_r", (E * H, I))
    np.testing.assert_array_equal(decode_mx(q, sf, "row").reshape(E, H, I), oracle.mx_qdq(W2, axis=2))
    W13 = inp.f64("W13")
    q, sf = _mxview(L, "w13_r", (E * 2 * I, H))
    dq = decode_mx(q, sf, "row").reshape(E, 2 * I // 128, 2, 64, H)     # blocks of [64 gate | 64 up]
    gate = dq[:, :, 0].reshape(E, I, H)
    up = dq[:, :, 1].reshape(E, I, H)
    ref = oracle.mx_qdq(W13, axis=2)
    np.testing.assert_array_equal(gate, ref[:, :I])
    np.testing.assert_array_equal(up, ref[:, I:])
    q, sf = _mxview(L, "w13_c", (E * 2 * I, H))
    np.testing.assert_array_equal(decode_mx(q, sf, "col").reshape(E, 2 * I, H), oracle.mx_qdq(W13, axis=1))


@pytest.mark.parametrize("name", list(SMALL))
def test_forward(cuda_lib, name):
    inp = gen.make_inputs(SMALL[name])
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.fwd()
    torch.cuda.synchronize()
    assert L.status() == 0
    y_ref = oracle.forward(*_args(inp), mxfp8=True)
    err = rel_fro(f64(L.y), y_ref)
    assert err < TOL, err
    assert max_row_rel(f64(L.y), y_ref) < ROW_TOL
    # and it is an MXFP8 result: closer to the quantised oracle than to the BF16 one
    assert err < rel_fro(f64(L.y), oracle.forward(*_args(inp)))


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("reuse", [False, True])
def test_backward(cuda_lib, name, reuse):
    inp = gen.make_inputs(SMALL[name])
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    flags = 0
    if reuse:
        L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
        flags = cuda_lib.MOE_FLAG_REUSE_FWD | cuda_lib.MOE_FLAG_REUSE_WEIGHTS
    L.bwd(flags=flags)
    torch.cuda.synchronize()
    assert L.status() == 0
    ref = oracle.backward(inp.f64("dy"), *_args(inp), mxfp8=True)
    for got, n in ((L.dx, "dx"), (L.dW13, "dW13"), (L.dW2, "dW2"), (L.dtw, "dtopk_w")):
        err = rel_fro(f64(got), ref[n])
        assert err < TOL, (n, err)
        if n != "dtopk_w":
            assert max_row_rel(f64(got), ref[n]) < ROW_TOL, (n, max_row_rel(f64(got), ref[n]))


def test_weight_reuse_is_exact_and_checked(cuda_lib):
    inp = gen.make_inputs(SMALL["medium"])
    A = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    A.fwd()
    A.bwd()
    B = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    with pytest.raises(cuda_lib.MoeError) as ei:
        B.fwd(flags=cuda_lib.MOE_FLAG_REUSE_WEIGHTS)     # nothing quantised on this scratch yet
    assert ei.value.code == cuda_lib.ERR["MOE_ERR_STATE"]
    B.fwd()
    B.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU | cuda_lib.MOE_FLAG_REUSE_WEIGHTS)
    B.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD | cuda_lib.MOE_FLAG_REUSE_WEIGHTS)
    torch.cuda.synchronize()
    for a, b in ((A.y, B.y), (A.dx, B.dx), (A.dW13, B.dW13), (A.dW2, B.dW2), (A.dtw, B.dtw)):
        assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["qwen3_30b_a3b_mxfp8", "qwen3_235b_a22b_mxfp8"])
def test_full_size_sampled(cuda_lib, name):
    cfg = gen.CONFIGS[name]
    inp = gen.make_inputs(cfg)
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.fwd()
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU | cuda_lib.MOE_FLAG_REUSE_WEIGHTS)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD | cuda_lib.MOE_FLAG_REUSE_WEIGHTS)
    torch.cuda.synchronize()
    assert L.status() == 0
    rng = np.random.default_rng(1)
    toks = np.sort(rng.choice(cfg.T, 8, replace=False))
    x, dy, W13, W2 = inp.f32("x"), inp.f32("dy"), inp.f32("W13"), inp.f32("W2")
    ti = torch.from_numpy(toks).cuda()
    y_s = oracle.forward_tokens(x, inp.topk_idx, inp.topk_w, W13, W2, toks, mxfp8=True)
    assert rel_fro(f64(L.y[ti]), y_s) < TOL
    dx_s, dtw_s = oracle.backward_tokens(dy, x, inp.topk_idx, inp.topk_w, W13, W2, toks, mxfp8=True)
    assert rel_fro(f64(L.dx[ti]), dx_s) < TOL
    assert rel_fro(f64(L.dtw[ti]), dtw_s) < TOL
    experts = [0, int(rng.integers(cfg.E))]
    for e, (a13, a2) in zip(experts, oracle.wgrad_experts(dy, x, inp.topk_idx, inp.topk_w, W13, W2, experts,
                                                          mxfp8=True)):
        assert rel_fro(f64(L.dW13[e]), a13) < TOL, e
        assert rel_fro(f64(L.dW2[e]), a2) < TOL, e
    for t in (L.y, L.dx, L.dW13, L.dW2, L.dtw):
        assert torch.isfinite(t).all()


def test_fused_epilogue_copies(cuda_lib):
    """The E4M3 copies the GEMM epilogues emit (h along I; [dg|du] along 2I and along the tokens;
    w h along the tokens) decode to the oracle's quantise-dequantise of the same quantities.
    The epilogues quantise fp32 values and the oracle fp64 ones, so a near-tie can round the
    other way (one E4M3 step, about 8%, on a few per cent of the values): compared in relative
    Frobenius norm against the MXFP8 bound."""
    inp = gen.make_inputs(SMALL["medium"])
    cfg = inp.cfg
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD | cuda_lib.MOE_FLAG_REUSE_WEIGHTS)
    torch.cuda.synchronize()
    assert L.status() == 0
    I, R = cfg.I, L.rows()
    r, prow = _padded_rows(L, inp)
    ref = oracle.backward(inp.f64("dy"), *_args(inp), mxfp8=True, keep=True)
    h = ref["fwd"]["h"]
    q, sf = _mxview(L, "h_r", (R, I))
    assert rel_fro(decode_mx(q, sf, "row")[prow], oracle.mx_qdq(h, axis=1)) < TOL
    q, sf = _mxview(L, "dg_r", (R, 2 * I))
    assert rel_fro(decode_mx(q, sf, "row")[prow], oracle.mx_qdq(ref["dG"], axis=1)) < TOL
    q, sf = _mxview(L, "dg_c", (R, 2 * I))
    assert rel_fro(decode_mx(q, sf, "col")[prow], oracle.mx_qdq_segments(ref["dG"], r["off"])) < TOL
    q, sf = _mxview(L, "hw_c", (R, I))
    assert rel_fro(decode_mx(q, sf, "col")[prow], oracle.mx_qdq_segments(ref["Hw"], r["off"])) < TOL


# ---------------------------------------------------------------- edge cases in both block-scaled modes
def _edge_inputs(case, precision):
    import dataclasses
    mk = lambda **kw: dataclasses.replace(gen.custom_config(**kw), precision=precision)   # noqa: E731
    if case == "one_token":
        return gen.make_inputs(mk(T=1, H=256, I=128, E=8, k=2, seed=31))
    if case == "all_on_one_expert":
        inp = gen.make_inputs(mk(T=300, H=256, I=128, E=8, k=1, seed=32))
        inp.topk_idx = np.full((300, 1), 5, dtype=np.int32)
        return inp
    if case == "empty_experts":
        inp = gen.make_inputs(mk(T=400, H=256, I=256, E=16, k=2, seed=33))
        inp.topk_idx = np.ascontiguousarray(np.stack([np.arange(400) % 3, 7 + np.arange(400) % 2], 1).astype(np.int32))
        return inp
    if case == "single_expert_top1":
        return gen.make_inputs(mk(T=200, H=256, I=128, E=1, k=1, seed=34))
    if case == "max_experts":   # 1024 experts, about four rows each, some idle
        return gen.make_inputs(mk(T=512, H=256, I=128, E=1024, k=8, seed=38))
    return gen.make_inputs(mk(T=20, H=512, I=256, E=4, k=2, seed=35))     # fewer rows than a tile


# (the 1024-expert case runs in MXFP8 only: its fp64 oracle takes about half a minute, and
# fp8_bwd runs the same block-scaled backward kernels)
@pytest.mark.parametrize("case,precision", [(c, p) for c in ("one_token", "all_on_one_expert", "empty_experts",
                                                             "single_expert_top1", "fewer_rows_than_a_tile",
                                                             "max_experts")
                                            for p in ("mxfp8", "fp8_bwd") if (c, p) != ("max_experts", "fp8_bwd")])
def test_edge_cases_block_scaled(cuda_lib, case, precision):
    inp = _edge_inputs(case, precision)
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.fwd()
    L.bwd()
    torch.cuda.synchronize()
    assert L.status() == 0
    mode = {"mxfp8": True} if precision == "mxfp8" else {"fp8_bwd": True}
    y = oracle.forward(*_args(inp), mxfp8=precision == "mxfp8")
    ref = oracle.backward(inp.f64("dy"), *_args(inp), **mode)
    assert rel_fro(f64(L.y), y) < TOL
    for got, n in ((L.dx, "dx"), (L.dW13, "dW13"), (L.dW2, "dW2"), (L.dtw, "dtopk_w")):
        if np.linalg.norm(ref[n]) == 0:
            assert torch.all(got == 0), n
        else:
            assert rel_fro(f64(got), ref[n]) < TOL, (n, rel_fro(f64(got), ref[n]))
    if case in ("empty_experts", "max_experts"):
        idle = sorted(set(range(inp.cfg.E)) - set(np.unique(inp.topk_idx).tolist()))
        assert torch.all(L.dW13[idle] == 0) and torch.all(L.dW2[idle] == 0)


@pytest.mark.parametrize("precision", ["mxfp8", "fp8_bwd"])
def test_zero_tokens_block_scaled(cuda_lib, precision):
    import dataclasses
    inp = gen.make_inputs(dataclasses.replace(gen.custom_config(T=0, H=256, I=128, E=8, k=2, seed=36),
                                              precision=precision))
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.float32)
    L.fwd()
    L.bwd()
    torch.cuda.synchronize()
    assert torch.all(L.dW13 == 0) and torch.all(L.dW2 == 0)


@pytest.mark.parametrize("case", ["medium", "empty_experts"])
def test_backward_bf16_weight_gradients(cuda_lib, case):
    """A caller may take dW13, dW2 in bf16 (reading 13: the caller's choice of dtype): the drained
    128 x 256 weight-gradient tiles then store bf16 rows, and experts without rows get zeros."""
    inp = gen.make_inputs(SMALL["medium"]) if case == "medium" else _edge_inputs("empty_experts", "mxfp8")
    L = DeviceLayer(cuda_lib, inp, wgrad_dtype=torch.bfloat16)
    L.fwd(flags=cuda_lib.MOE_FLAG_SAVE_GU)
    L.bwd(flags=cuda_lib.MOE_FLAG_REUSE_FWD | cuda_lib.MOE_FLAG_REUSE_WEIGHTS)
    torch.cuda.synchronize()
    assert L.status() == 0
    ref = oracle.backward(inp.f64("dy"), *_args(inp), mxfp8=True)
    for got, n in ((L.dW13, "dW13"), (L.dW2, "dW2")):
        assert got.dtype == torch.bfloat16
        assert rel_fro(f64(got), ref[n]) < TOL, (n, rel_fro(f64(got), ref[n]))
    if case == "empty_experts":
        idle = sorted(set(range(inp.cfg.E)) - set(np.unique(inp.topk_idx).tolist()))
        assert idle and torch.all(L.dW13[idle] == 0) and torch.all(L.dW2[idle] == 0)
