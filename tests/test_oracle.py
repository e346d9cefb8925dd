"""Pins of the fp64 oracle against things other than itself (CPU only).

* routing: numpy's stable argsort and the bincount/cumsum definitions of counts and offsets;
* forward: a dense form where every token runs every expert with weight 0 off its top-k, written
  with einsum; and the k = 1, E = 1 special case, a plain SwiGLU MLP;
* backward: torch float64 autograd of the dense form, and central finite differences;
* MXFP8: the E4M3 code table decoded from its bit fields, torch's float8_e4m3fn cast, and the
  OCP MX shared-exponent rule on hand-built blocks.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen


def _small_cfg(T=64, H=32, I=16, E=6, k=2, routing="uniform", seed=7):
    return gen.custom_config(T=T, H=H, I=I, E=E, k=k, routing=routing, seed=seed)


def _f64(inp):
    return (inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2"), inp.f64("dy"))


# ---------------------------------------------------------------- routing
@pytest.mark.parametrize("cfg", [
    _small_cfg(), _small_cfg(T=300, E=16, k=4, seed=3), _small_cfg(T=500, E=12, k=8, routing="zipf", seed=5),
    gen.CONFIGS["tiny"],
])
def test_route_matches_stable_argsort(cfg):
    idx, _ = gen.routing(cfg)
    r = oracle.route(idx, cfg.E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(r["perm"], np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(r["cnt"], np.bincount(flat, minlength=cfg.E))
    np.testing.assert_array_equal(r["off"], np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=cfg.E))]))


def test_route_invariants():
    cfg = _small_cfg(T=777, E=32, k=8, routing="zipf", seed=11)
    idx, _ = gen.routing(cfg)
    r = oracle.route(idx, cfg.E)
    S = cfg.S
    assert r["cnt"].sum() == S and r["off"][-1] == S and r["off"][0] == 0
    assert sorted(r["perm"].tolist()) == list(range(S))
    np.testing.assert_array_equal(r["inv"][r["perm"]], np.arange(S))
    flat = idx.reshape(-1)
    assert np.all(np.diff(flat[r["perm"]]) >= 0)
    for e in range(cfg.E):
        grp = r["perm"][r["off"][e]:r["off"][e + 1]]
        assert np.all(np.diff(grp) > 0)          # slots ascend inside each group (stability)
        assert np.all(flat[grp] == e)


def test_route_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0, 5]]), 5)


def test_permute_unpermute_identity():
    cfg = _small_cfg(T=200, E=10, k=3, seed=2)
    inp = gen.make_inputs(cfg)
    x = inp.f64("x")
    r = oracle.route(inp.topk_idx, cfg.E)
    Xp = oracle.permute_rows(x, r["perm"], cfg.k)
    w = inp.topk_w.astype(np.float64)
    w = w / w.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(oracle.unpermute_sum(Xp, r["inv"], cfg.T, cfg.k, w), x, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.unpermute_sum(Xp, r["inv"], cfg.T, cfg.k), cfg.k * x, rtol=1e-13)


# ---------------------------------------------------------------- dense brute-force forms
def _dense_gate(idx, w, T, E):
    D = np.zeros((T, E))
    for t in range(T):
        for j in range(idx.shape[1]):
            D[t, idx[t, j]] += w[t, j]
    return D


def _dense_forward_np(x, idx, w, W13, W2):
    T, E, I = x.shape[0], W13.shape[0], W13.shape[1] // 2
    G = np.einsum("th,eih->tei", x, W13[:, :I])
    U = np.einsum("th,eih->tei", x, W13[:, I:])
    Hh = G / (1.0 + np.exp(-G)) * U
    O = np.einsum("tei,ehi->teh", Hh, W2)
    return np.einsum("te,teh->th", _dense_gate(idx, w, T, E), O)


def _dense_torch_grads(x, idx, w, W13, W2, dy):
    T, E, I = x.shape[0], W13.shape[0], W13.shape[1] // 2
    tx = torch.tensor(x, requires_grad=True)
    tw = torch.tensor(w, requires_grad=True)
    t13 = torch.tensor(W13, requires_grad=True)
    t2 = torch.tensor(W2, requires_grad=True)
    D = torch.zeros(T, E, dtype=torch.float64).scatter_add(1, torch.tensor(idx, dtype=torch.int64), tw)
    G = torch.einsum("th,eih->tei", tx, t13[:, :I])
    U = torch.einsum("th,eih->tei", tx, t13[:, I:])
    y = torch.einsum("te,teh->th", D, torch.einsum("tei,ehi->teh", torch.nn.functional.silu(G) * U, t2))
    (y * torch.tensor(dy)).sum().backward()
    return {"y": y.detach().numpy(), "dx": tx.grad.numpy(), "dtopk_w": tw.grad.numpy(),
            "dW13": t13.grad.numpy(), "dW2": t2.grad.numpy()}


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


@pytest.mark.parametrize("cfg", [gen.CONFIGS["tiny"], _small_cfg(T=97, E=5, k=3, seed=9),
                                 _small_cfg(T=120, E=9, k=4, routing="zipf", seed=4)])
def test_forward_matches_dense_all_experts(cfg):
    x, idx, w, W13, W2, _ = _f64(gen.make_inputs(cfg))
    y = oracle.forward(x, idx, w, W13, W2)
    assert _rel(y, _dense_forward_np(x, idx, w, W13, W2)) < 1e-12


def test_single_expert_top1_is_swiglu_mlp():
    rng = np.random.default_rng(0)
    T, H, I = 13, 24, 10
    x = rng.standard_normal((T, H)); W1 = rng.standard_normal((I, H)); W3 = rng.standard_normal((I, H))
    Wd = rng.standard_normal((H, I)); w = rng.random((T, 1))
    y = oracle.forward(x, np.zeros((T, 1), dtype=np.int32), w, np.concatenate([W1, W3])[None], Wd[None])
    a = x @ W1.T
    ref = w * ((a / (1.0 + np.exp(-a)) * (x @ W3.T)) @ Wd.T)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("cfg", [gen.CONFIGS["tiny"], _small_cfg(T=150, E=7, k=3, seed=21),
                                 _small_cfg(T=90, E=10, k=5, routing="zipf", seed=8)])
def test_backward_matches_torch_autograd(cfg):
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    got = oracle.backward(dy, x, idx, w, W13, W2)
    ref = _dense_torch_grads(x, idx, w, W13, W2, dy)
    for name in ("dx", "dW13", "dW2", "dtopk_w"):
        assert _rel(got[name], ref[name]) < 1e-11, name


def test_backward_matches_central_differences():
    cfg = _small_cfg(T=6, H=8, I=4, E=3, k=2, seed=1)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    g = oracle.backward(dy, x, idx, w, W13, W2)
    loss = lambda x_, w_, a_, b_: float(np.sum(dy * oracle.forward(x_, idx, w_, a_, b_)))
    rng = np.random.default_rng(5)
    eps = 1e-6
    for name, arr, pos in (("dx", x, 0), ("dtopk_w", w, 1), ("dW13", W13, 2), ("dW2", W2, 3)):
        for _ in range(6):
            i = tuple(int(rng.integers(0, n)) for n in arr.shape)
            args_p = [x.copy(), w.copy(), W13.copy(), W2.copy()]
            args_m = [x.copy(), w.copy(), W13.copy(), W2.copy()]
            args_p[pos][i] += eps
            args_m[pos][i] -= eps
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[name][i]) <= 1e-7 * max(1.0, abs(fd)), (name, i, fd, g[name][i])


def test_empty_expert_has_zero_weight_grad():
    cfg = _small_cfg(T=40, E=8, k=2, seed=3)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    idx = np.where(idx == 5, 6, idx).astype(np.int32)
    idx[:, 1] = np.where(idx[:, 0] == idx[:, 1], (idx[:, 1] + 1) % 5, idx[:, 1])
    assert not np.any(idx == 5)
    g = oracle.backward(dy, x, idx, w, W13, W2)
    assert np.all(g["dW13"][5] == 0) and np.all(g["dW2"][5] == 0)
    ref = _dense_torch_grads(x, idx, w, W13, W2, dy)
    assert _rel(g["dW13"], ref["dW13"]) < 1e-11


def test_sampled_forms_agree_with_full():
    cfg = _small_cfg(T=80, H=32, I=16, E=6, k=3, seed=12)
    inp = gen.make_inputs(cfg)
    x, idx, w, W13, W2, dy = _f64(inp)
    y = oracle.forward(x, idx, w, W13, W2)
    g = oracle.backward(dy, x, idx, w, W13, W2)
    toks = [0, 17, 79]
    np.testing.assert_allclose(oracle.forward_tokens(x, idx, w, W13, W2, toks), y[toks], rtol=1e-11, atol=1e-12)
    dx, dtw = oracle.backward_tokens(dy, x, idx, w, W13, W2, toks)
    np.testing.assert_allclose(dx, g["dx"][toks], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dtw, g["dtopk_w"][toks], rtol=1e-11, atol=1e-12)
    for e, (a, b) in zip([1, 4], oracle.wgrad_experts(dy, x, idx, w, W13, W2, [1, 4])):
        np.testing.assert_allclose(a, g["dW13"][e], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(b, g["dW2"][e], rtol=1e-11, atol=1e-12)
    yq = oracle.forward(x, idx, w, W13, W2, mxfp8=True)
    np.testing.assert_allclose(oracle.forward_tokens(x, idx, w, W13, W2, toks, mxfp8=True), yq[toks],
                               rtol=1e-11, atol=1e-12)
    gq = oracle.backward(dy, x, idx, w, W13, W2, mxfp8=True)
    dxq, dtwq = oracle.backward_tokens(dy, x, idx, w, W13, W2, toks, mxfp8=True)
    np.testing.assert_allclose(dxq, gq["dx"][toks], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dtwq, gq["dtopk_w"][toks], rtol=1e-11, atol=1e-12)
    for e, (a, b) in zip([1, 4], oracle.wgrad_experts(dy, x, idx, w, W13, W2, [1, 4], mxfp8=True)):
        np.testing.assert_allclose(a, gq["dW13"][e], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(b, gq["dW2"][e], rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- planted mistakes must be caught
def test_pins_catch_a_planted_sign_error(monkeypatch):
    cfg = _small_cfg(T=30, E=4, k=2, seed=6)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    ref = _dense_torch_grads(x, idx, w, W13, W2, dy)
    monkeypatch.setattr(oracle.moe_oracle, "sigmoid", lambda z: 1.0 / (1.0 + np.exp(z)))
    got = oracle.backward(dy, x, idx, w, W13, W2)
    assert _rel(got["dx"], ref["dx"]) > 1e-3


def test_pins_catch_a_planted_unstable_sort(monkeypatch):
    cfg = _small_cfg(T=50, E=4, k=2, seed=6)
    idx, _ = gen.routing(cfg)
    good = oracle.route(idx, cfg.E)["perm"]
    flat = idx.reshape(-1)
    assert not np.array_equal(np.argsort(flat, kind="quicksort")[::-1], good)


# ---------------------------------------------------------------- MXFP8 quantiser
def _e4m3_code_values():
    """All finite E4M3 values decoded from the bit fields: sign, 4 exponent bits (bias 7),
    3 mantissa bits; exponent field 0 is subnormal; S.1111.111 is NaN."""
    vals = []
    for code in range(256):
        s, ex, m = code >> 7, (code >> 3) & 0xF, code & 7
        if ex == 0xF and m == 7:
            continue
        v = (m / 8.0) * 2.0 ** -6 if ex == 0 else (1 + m / 8.0) * 2.0 ** (ex - 7)
        vals.append(-v if s else v)
    return np.array(vals)


def test_e4m3_grid_round_trips():
    vals = _e4m3_code_values()
    assert len(vals) == 254 and vals.max() == 448.0 and np.min(vals[vals > 0]) == 2.0 ** -9
    np.testing.assert_array_equal(oracle.e4m3_round(vals), vals)


def test_e4m3_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.uniform(-3, 2.3, 200000),
                        rng.uniform(-448, 448, 50000), _e4m3_code_values() * 1.0625])
    v = v[np.abs(v) <= 448.0].astype(np.float32).astype(np.float64)
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_round(v), ref)
    assert oracle.e4m3_round(np.array([460.0, -1000.0]))[0] == 448.0
    assert oracle.e4m3_round(np.array([-1000.0]))[0] == -448.0


def test_mx_exponent_rule_on_hand_built_blocks():
    # amax = 1.0 -> floor(log2) = 0 -> shared exponent -8, elements scaled by 256
    np.testing.assert_array_equal(oracle.mx_block_exponent(np.array([1.0, 1.99, 2.0, 448.0, 0.0])),
                                  [-8, -8, -7, 0, -127])
    blk = np.zeros(32); blk[0] = 1.0; blk[1] = 1.0 / 256; blk[2] = 1.0 / 4096; blk[3] = 1.7
    q = oracle.mx_qdq(blk[None], axis=1)[0]
    # 1.7 * 256 = 435.2 -> nearest E4M3 is 448 (spacing 32 above 256): 448/256 = 1.75
    np.testing.assert_allclose(q[:4], [1.0, 1.0 / 256, 1.0 / 4096, 1.75])
    # a block whose scaled max exceeds 448 saturates: amax 1.99 * 256 = 509 -> 448
    assert oracle.mx_qdq(np.array([[1.99] + [0.0] * 31]), axis=1)[0, 0] == 448.0 / 256


def test_mx_qdq_axis_and_segments():
    rng = np.random.default_rng(1)
    a = rng.standard_normal((64, 96))
    q0 = oracle.mx_qdq(a, axis=0)
    q1 = oracle.mx_qdq(a, axis=1)
    np.testing.assert_array_equal(q0, oracle.mx_qdq(a.T, axis=1).T)
    np.testing.assert_array_equal(oracle.mx_qdq(q1, axis=1), q1)        # idempotent
    rel = np.abs(q1 - a) / np.maximum(np.abs(a), 1e-30)
    amax = np.repeat(np.abs(a).reshape(64, 3, 32).max(axis=2), 32, axis=1)
    scaled = np.abs(a) / np.ldexp(1.0, oracle.mx_block_exponent(amax))
    normal = (scaled >= 2.0 ** -6) & (scaled <= 448.0)
    assert rel[normal].max() <= 2.0 ** -4 + 1e-12        # 3 mantissa bits: half a step
    assert rel[scaled > 448.0].max() <= 0.125            # saturation of (448, 512) to 448
    starts = np.array([0, 10, 10, 50, 64])
    s = oracle.mx_qdq_segments(a, starts)
    np.testing.assert_array_equal(s[10:50], oracle.mx_qdq(a[10:50], axis=0))
    padded = np.concatenate([a[50:64], np.zeros((18, 96))])
    np.testing.assert_array_equal(s[50:64], oracle.mx_qdq(padded, axis=0)[:14])


def test_mxfp8_quantisation_points_follow_the_contraction_axes(monkeypatch):
    """Every quantised GEMM operand is blocked along that GEMM's contraction axis."""
    cfg = _small_cfg(T=40, H=64, I=96, E=3, k=2, seed=14)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    calls = []
    in_seg = []
    real, real_seg = oracle.moe_oracle.mx_qdq, oracle.moe_oracle.mx_qdq_segments

    def rec(a, axis, fmt="e4m3"):
        assert fmt == "e4m3"
        if not in_seg:
            calls.append(("ax", np.shape(a), axis))
        return real(a, axis)

    def rec_seg(a, st):
        calls.append(("seg", np.shape(a), 0))
        in_seg.append(1)
        try:
            return real_seg(a, st)
        finally:
            in_seg.pop()
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq", rec)
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq_segments", rec_seg)
    oracle.backward(dy, x, idx, w, W13, W2, mxfp8=True)
    H, I, S = 64, 96, 80
    lengths = {c[1][c[2]] if c[0] == "ax" else "tokens" for c in calls}
    assert lengths <= {H, I, 2 * I, "tokens"}
    seen = {(c[0], c[1], c[2]) for c in calls}
    assert ("ax", (S, H), 1) in seen                   # X_perm and dY_perm along H
    assert ("ax", (H, I), 1) in seen                   # W2 along I for the forward down GEMM
    assert ("ax", (H, I), 0) in seen                   # W2 along H for the backward dgrad
    assert ("ax", (2 * I, H), 0) in seen               # W13 along 2I for the backward dgrad
    assert ("ax", (I, H), 1) in seen                   # W13 gate/up along H for the forward
    assert sum(1 for c in calls if c[0] == "seg") == 4  # dY, Hw, dG, X along tokens per expert


def test_mxfp8_with_identity_quantiser_equals_bf16_path(monkeypatch):
    cfg = _small_cfg(T=48, H=32, I=32, E=4, k=2, seed=15)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    ref = oracle.backward(dy, x, idx, w, W13, W2)
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq", lambda a, axis, fmt="e4m3": np.asarray(a, dtype=np.float64))
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq_segments", lambda a, st: np.asarray(a, dtype=np.float64))
    monkeypatch.setattr(oracle.moe_oracle, "_stored_bf16", lambda a: np.asarray(a, dtype=np.float64))
    got = oracle.backward(dy, x, idx, w, W13, W2, mxfp8=True)
    for k_ in ("dx", "dW13", "dW2", "dtopk_w"):
        np.testing.assert_allclose(got[k_], ref[k_], rtol=1e-13, atol=1e-13)


def test_mxfp8_error_is_at_quantisation_scale():
    cfg = gen.CONFIGS["tiny"]
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    y = oracle.forward(x, idx, w, W13, W2)
    yq = oracle.forward(x, idx, w, W13, W2, mxfp8=True)
    e = _rel(yq, y)
    assert 2e-3 < e < 8e-2


# ---------------------------------------------------------------- fp8_bwd: BF16 forward, MXFP8 backward
def _record_quantiser_calls(monkeypatch):
    calls, in_seg = [], []
    real, real_seg = oracle.moe_oracle.mx_qdq, oracle.moe_oracle.mx_qdq_segments

    def rec(a, axis, fmt="e4m3"):
        assert fmt == "e4m3"
        if not in_seg:
            calls.append(("ax", np.shape(a), axis))
        return real(a, axis)

    def rec_seg(a, st):
        calls.append(("seg", np.shape(a), 0))
        in_seg.append(1)
        try:
            return real_seg(a, st)
        finally:
            in_seg.pop()
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq", rec)
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq_segments", rec_seg)
    return calls


def test_fp8_bwd_quantises_only_the_backward_contractions(monkeypatch):
    """fp8_bwd: the forward's X, W13 (along H), h and W2 (along I) stay exact; dY along H, W2 along
    H, W13 and [dg|du] along 2I and the four weight-gradient operands along tokens are quantised."""
    cfg = _small_cfg(T=40, H=64, I=96, E=3, k=2, seed=14)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    calls = _record_quantiser_calls(monkeypatch)
    oracle.backward(dy, x, idx, w, W13, W2, fp8_bwd=True)
    H, I, S = 64, 96, 80
    ax = [c for c in calls if c[0] == "ax"]
    assert sum(1 for c in ax if c[1] == (S, H) and c[2] == 1) == 1       # dY_perm only, not X_perm
    assert not any(c[1] == (H, I) and c[2] == 1 for c in ax)             # no forward W2 blocks
    assert not any(c[1] == (I, H) and c[2] == 1 for c in ax)             # no forward W13 blocks
    assert any(c[1] == (H, I) and c[2] == 0 for c in ax)                 # W2 along H (dgrad)
    assert any(c[1] == (2 * I, H) and c[2] == 0 for c in ax)             # W13 along 2I (dgrad)
    assert any(len(c[1]) == 2 and c[1][1] == 2 * I and c[2] == 1 for c in ax)   # [dg|du] along 2I
    assert not any(len(c[1]) == 2 and c[1][1] == I and c[1][0] != H and c[2] == 1 for c in ax)  # no h
    assert sum(1 for c in calls if c[0] == "seg") == 4


def test_fp8_bwd_with_identity_quantiser_equals_bf16_path(monkeypatch):
    cfg = _small_cfg(T=48, H=32, I=32, E=4, k=2, seed=15)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    ref = oracle.backward(dy, x, idx, w, W13, W2)
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq", lambda a, axis, fmt="e4m3": np.asarray(a, dtype=np.float64))
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq_segments", lambda a, st: np.asarray(a, dtype=np.float64))
    monkeypatch.setattr(oracle.moe_oracle, "_stored_bf16", lambda a: np.asarray(a, dtype=np.float64))
    got = oracle.backward(dy, x, idx, w, W13, W2, fp8_bwd=True)
    for k_ in ("dx", "dW13", "dW2", "dtopk_w"):
        np.testing.assert_allclose(got[k_], ref[k_], rtol=1e-13, atol=1e-13)


def test_fp8_bwd_sampled_forms_agree_with_full():
    cfg = _small_cfg(T=80, H=32, I=16, E=6, k=3, seed=12)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    g = oracle.backward(dy, x, idx, w, W13, W2, fp8_bwd=True)
    toks = [0, 17, 79]
    dx, dtw = oracle.backward_tokens(dy, x, idx, w, W13, W2, toks, fp8_bwd=True)
    np.testing.assert_allclose(dx, g["dx"][toks], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dtw, g["dtopk_w"][toks], rtol=1e-11, atol=1e-12)
    for e, (a, b) in zip([1, 4], oracle.wgrad_experts(dy, x, idx, w, W13, W2, [1, 4], fp8_bwd=True)):
        np.testing.assert_allclose(a, g["dW13"][e], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(b, g["dW2"][e], rtol=1e-11, atol=1e-12)


def test_fp8_bwd_error_is_at_quantisation_scale_and_differs_from_mxfp8():
    cfg = gen.CONFIGS["tiny"]
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    ref = oracle.backward(dy, x, idx, w, W13, W2)
    got = oracle.backward(dy, x, idx, w, W13, W2, fp8_bwd=True)
    mx = oracle.backward(dy, x, idx, w, W13, W2, mxfp8=True)
    for k_ in ("dx", "dW13", "dW2", "dtopk_w"):
        assert 1e-3 < _rel(got[k_], ref[k_]) < 8e-2, k_
        assert _rel(got[k_], mx[k_]) > 1e-4, k_       # the forward differs (exact vs quantised)


# ---------------------------------------------------------------- router (the step before the layer)
def test_router_selects_the_largest_logits_ties_to_lower_index():
    rng = np.random.default_rng(31)
    L = np.round(rng.standard_normal((200, 24)) * 2) / 2          # many ties
    idx, w = oracle.router_forward(L.astype(np.float32), 5)
    for t in range(200):
        sel = list(idx[t])
        assert len(set(sel)) == 5
        rest = [e for e in range(24) if e not in sel]
        assert L[t, sel].min() >= L[t, rest].max()
        assert all(L[t, sel[j]] >= L[t, sel[j + 1]] for j in range(4))   # descending
        for j in range(4):                                              # equal logits: lower index first
            if L[t, sel[j]] == L[t, sel[j + 1]]:
                assert sel[j] < sel[j + 1]
        # a tie across the cut keeps the lower indices
        cut = L[t, sel[-1]]
        tied = [e for e in range(24) if L[t, e] == cut]
        kept = [e for e in sel if L[t, e] == cut]
        assert kept == tied[:len(kept)]


def test_router_weights_are_the_softmax_of_the_selected_logits():
    from scipy.special import softmax
    rng = np.random.default_rng(32)
    L = rng.standard_normal((50, 16)).astype(np.float32)
    idx, w = oracle.router_forward(L, 16)                         # k = E: the full softmax
    full = softmax(L.astype(np.float64), axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(full, idx.astype(np.int64), 1), rtol=1e-13)
    idx, w = oracle.router_forward(L, 4)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-14)
    sel = np.take_along_axis(L.astype(np.float64), idx.astype(np.int64), 1)
    np.testing.assert_allclose(w[:, 1:] / w[:, :1], np.exp(sel[:, 1:] - sel[:, :1]), rtol=1e-12)


def test_router_backward_matches_finite_differences_and_autograd():
    import torch
    rng = np.random.default_rng(33)
    T, E, k = 6, 12, 3
    # well-separated logits: a step of 1e-6 never changes the selection
    L = np.stack([rng.permutation(E) * 0.5 + rng.uniform(-0.1, 0.1) for _ in range(T)])
    dw = rng.standard_normal((T, k))
    idx, w = oracle.router_forward(L, k)
    dl = oracle.router_backward(idx, w, dw, E)

    def loss(LL):
        i2, w2 = oracle.router_forward(LL, k)
        assert np.array_equal(i2, idx)
        return float((w2 * dw).sum())
    h = 1e-6
    for t in range(T):
        for e in range(E):
            P, M = L.copy(), L.copy()
            P[t, e] += h
            M[t, e] -= h
            assert abs((loss(P) - loss(M)) / (2 * h) - dl[t, e]) < 1e-8
    lt = torch.tensor(L, requires_grad=True)
    sel = torch.gather(lt, 1, torch.tensor(idx, dtype=torch.int64))
    (torch.softmax(sel, 1) * torch.tensor(dw)).sum().backward()
    np.testing.assert_allclose(dl, lt.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_stored_bf16_rounds_to_nearest_even():
    """The bf16 storage of the saved pre-activations against torch's own float32 -> bfloat16 cast,
    on random values and on exact ties."""
    import torch
    rng = np.random.default_rng(34)
    a = np.concatenate([rng.standard_normal(100000) * 10 ** rng.uniform(-3, 3, 100000),
                        # exact ties between two bf16 neighbours, both parities
                        (np.arange(1, 2001, dtype=np.float64) * 2 + 1) * 2.0 ** -8])
    got = oracle.moe_oracle._stored_bf16(a)
    ref = torch.tensor(a.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)


def test_quantised_backward_reads_bf16_stored_pre_activations(monkeypatch):
    """With identity quantisers the only difference left between the fp8_bwd and the BF16 backward
    is the bf16 storage of g and u: small, and gone when the storage is exact too."""
    cfg = _small_cfg(T=48, H=32, I=32, E=4, k=2, seed=15)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    ref = oracle.backward(dy, x, idx, w, W13, W2)
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq", lambda a, axis, fmt="e4m3": np.asarray(a, dtype=np.float64))
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq_segments", lambda a, st: np.asarray(a, dtype=np.float64))
    got = oracle.backward(dy, x, idx, w, W13, W2, fp8_bwd=True)
    for k_ in ("dx", "dW13", "dW2", "dtopk_w"):
        assert 1e-6 < _rel(got[k_], ref[k_]) < 1e-2, k_


# ---------------------------------------------------------------- MXFP4 weights (FP8 x FP4 forward)
def test_e2m1_grid_round_trips_ties_to_even_and_saturates():
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    for g in np.concatenate([grid, -grid]):
        assert oracle.e2m1_round(np.array([g]))[0] == g
    mids = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}   # ties to the even code
    for v, q in mids.items():
        assert oracle.e2m1_round(np.array([v]))[0] == q, v
        assert oracle.e2m1_round(np.array([-v]))[0] == -q, v
    assert oracle.e2m1_round(np.array([5.9, 7.0, 1e9]))[0] == 6.0
    assert np.all(oracle.e2m1_round(np.array([7.0, 1e9, -50.0])) == np.array([6.0, 6.0, -6.0]))


def test_mxfp4_block_exponent_on_hand_built_blocks():
    b = np.zeros((1, 32))
    b[0, :3] = [6.0, 1.0, -0.75]              # amax 6: exponent floor(log2 6) - 2 = 0, scale 1
    np.testing.assert_array_equal(oracle.mx_qdq(b, axis=1, fmt="e2m1")[0, :3], [6.0, 1.0, -1.0])
    b[0, :3] = [1.0, 0.3, 0.2]                # amax 1: exponent -2, scale 1/4: 0.3 -> 1.2 -> 1.0 -> 0.25
    np.testing.assert_allclose(oracle.mx_qdq(b, axis=1, fmt="e2m1")[0, :3], [1.0, 0.25, 0.25])
    b[0, :3] = [7.5, 7.0, 0.0]                # amax 7.5: exponent 0, 7.5 and 7 saturate to 6
    np.testing.assert_array_equal(oracle.mx_qdq(b, axis=1, fmt="e2m1")[0, :3], [6.0, 6.0, 0.0])


def test_fp8_fp4_forward_quantises_weights_to_e2m1_and_activations_to_e4m3(monkeypatch):
    cfg = _small_cfg(T=40, H=64, I=96, E=3, k=2, seed=14)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    calls = []
    real = oracle.moe_oracle.mx_qdq

    def rec(a, axis, fmt="e4m3"):
        calls.append((np.shape(a), axis, fmt))
        return real(a, axis, fmt)
    monkeypatch.setattr(oracle.moe_oracle, "mx_qdq", rec)
    oracle.forward(x, idx, w, W13, W2, fp8_fp4=True)
    H, I, S = 64, 96, 80
    assert ((S, H), 1, "e4m3") in calls                       # X_perm along H
    assert all(c[2] == "e2m1" for c in calls if c[0] in ((I, H), (H, I)))   # every weight block
    assert ((I, H), 1, "e2m1") in calls and ((H, I), 1, "e2m1") in calls
    assert any(c[0][1] == I and c[0][0] not in (H,) and c[2] == "e4m3" for c in calls)   # h along I


def test_fp8_fp4_identity_quantiser_and_sampled_form():
    cfg = _small_cfg(T=80, H=64, I=32, E=6, k=3, seed=12)
    x, idx, w, W13, W2, dy = _f64(gen.make_inputs(cfg))
    y = oracle.forward(x, idx, w, W13, W2, fp8_fp4=True)
    toks = [0, 17, 79]
    np.testing.assert_allclose(oracle.forward_tokens(x, idx, w, W13, W2, toks, fp8_fp4=True), y[toks],
                               rtol=1e-11, atol=1e-12)
    y_bf = oracle.forward(x, idx, w, W13, W2)
    assert 5e-2 < _rel(y, y_bf) < 4e-1      # E2M1 weights (one mantissa bit) through two GEMMs
    import unittest.mock as um
    with um.patch.object(oracle.moe_oracle, "mx_qdq", lambda a, axis, fmt="e4m3": np.asarray(a, dtype=np.float64)):
        np.testing.assert_allclose(oracle.forward(x, idx, w, W13, W2, fp8_fp4=True), y_bf, rtol=1e-13, atol=1e-13)


def test_e2m1_round_matches_brute_force_nearest_even():
    """e2m1_round against a brute force written from the format: the nearest of the eight
    magnitudes, a tie going to the code whose mantissa bit is 0, saturation at 6."""
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])      # codes 0..7, mantissa = code & 1
    rng = np.random.default_rng(11)
    mids = (mags[1:] + mags[:-1]) / 2
    v = np.concatenate([rng.uniform(0, 8, 200_000), mids, np.nextafter(mids, 0), np.nextafter(mids, 9),
                        mags, [6.5, 7.0, 100.0, 1e-30]])
    v = np.concatenate([v, -v])
    a = np.minimum(np.abs(v), 6.0)
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    odd = (np.arange(8) & 1).astype(bool)
    pick = np.where(cand.sum(axis=1) > 1, np.argmax(cand & ~odd[None, :], axis=1), np.argmax(cand, axis=1))
    expect = np.copysign(mags[pick], v)
    np.testing.assert_array_equal(oracle.e2m1_round(v), expect)
