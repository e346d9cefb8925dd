"""Plain, slow, fp64 reference of the MoE expert layer.  TEST INFRASTRUCTURE ONLY.

What the layer computes, as the pages describe it:

* Each token is routed to k of E experts with a routing weight; tokens are grouped by expert
  (per-expert counts, group offsets, a token reorder), every expert runs its own small matrix
  product on its group, and the expert outputs are aggregated back per token by routing weight
  (kongchang.com, "Prime Intellect推出Prime Mega MoE", section "为什么 MoE 训练特别需要融合内核",
  the grouped-GEMM explainer).
* The fused layer is expert-parallel dispatch, the two expert linear layers, SwiGLU, and combine
  (MarkTechPost, "Prime Intellect Releases Prime Mega MoE", section "How does the fused kernel
  work?").  The experts are gated and carry no bias (ic.work analysis, section
  "算子下沉时代的硬件死锁暗礁").  With every expert on one device, dispatch is a gather of token
  rows into expert order and combine is the weighted sum back to token order.
* Training needs the backward of the same layer, activation and weight gradients (MarkTechPost,
  "How does the fused kernel work?"; ic.work, section "从 3.11 倍到 1.32 倍的性能漏斗").

Readings where the pages are silent (each is also listed with the design notes):
  W13 is [E, 2I, H] with rows [0, I) the gate projection and rows [I, 2I) the up projection;
  SwiGLU is silu(g) * u with silu(z) = z * sigmoid(z), no clamp; the routing weight multiplies
  the expert output (after the down projection); the token reorder is stable by slot index
  s = t*k + j; the backward is that of the loss <dy, y>.

MXFP8 (OCP Microscaling v1.0, E4M3 elements, one E8M0 scale per 32 elements along the
contraction axis): the oracle quantises and dequantises each GEMM operand at the point where the
CUDA path feeds the block-scaled MMA, then computes in fp64.  The pages also name an fp8_bwd
precision, a BF16 forward with an FP8 backward (MarkTechPost, "Prime Intellect Releases Prime
Mega MoE", section "How does the fused kernel work?"); on Blackwell its FP8 is read as MXFP8, so
`fp8_bwd=True` keeps the forward operands exact and quantises only the four backward GEMMs'
operands, at the same points as the MXFP8 backward.  The shared exponent of a block is
floor(log2(amax)) - 8 (8 is the largest E4M3 exponent); elements are divided by 2^exp, rounded to
the nearest E4M3 value (ties to even) and saturated to +-448.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "route", "permute_rows", "unpermute_sum", "sigmoid", "silu",
    "e4m3_round", "e2m1_round", "mx_block_exponent", "mx_qdq", "mx_qdq_segments",
    "forward", "backward", "forward_tokens", "backward_tokens", "wgrad_experts",
    "router_forward", "router_backward",
]


# ----------------------------------------------------------------------------------------------
# routing bookkeeping: per-expert counts, group offsets, stable token reorder and its inverse
# ----------------------------------------------------------------------------------------------
def route(topk_idx: np.ndarray, E: int) -> dict:
    """Group the T*k slots by expert (counting sort, stable in slot order s = t*k + j).

    Returns cnt[E] (tokens per expert), off[E+1] (exclusive prefix of cnt: the group offsets),
    perm[S] (perm[p] = slot at sorted position p) and inv[S] (inv[perm[p]] = p).
    """
    flat = np.asarray(topk_idx).reshape(-1).astype(np.int64)
    S = flat.size
    if S and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    cnt = np.zeros(E, dtype=np.int64)
    for e in flat:
        cnt[e] += 1
    off = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        off[e + 1] = off[e] + cnt[e]
    perm = np.empty(S, dtype=np.int64)
    fill = off[:E].copy()
    for s in range(S):                       # walking slots in order keeps ties in slot order
        e = flat[s]
        perm[fill[e]] = s
        fill[e] += 1
    inv = np.empty(S, dtype=np.int64)
    inv[perm] = np.arange(S, dtype=np.int64)
    return {"cnt": cnt, "off": off, "perm": perm, "inv": inv}


def permute_rows(x: np.ndarray, perm: np.ndarray, k: int) -> np.ndarray:
    """Dispatch: row p of the result is the token of slot perm[p]."""
    return x[perm // k]


def unpermute_sum(rows: np.ndarray, inv: np.ndarray, T: int, k: int, weights=None) -> np.ndarray:
    """Combine: out[t] = sum_j weights[t, j] * rows[inv[t*k + j]] (unweighted if weights is None)."""
    out = np.zeros((T,) + rows.shape[1:], dtype=np.float64)
    for j in range(k):
        r = rows[inv[np.arange(T) * k + j]]
        out += r if weights is None else weights[:, j:j + 1] * r
    return out


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


# ----------------------------------------------------------------------------------------------
# MXFP8: E4M3 elements with one E8M0 power-of-two scale per block of 32
# ----------------------------------------------------------------------------------------------
E4M3_MAX = 448.0
E4M3_EMAX = 8          # exponent of the largest normal E4M3 value (448 = 1.75 * 2^8)
E4M3_EMIN = -6         # exponent of the smallest normal; subnormal spacing is 2^-9
MX_BLOCK = 32


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value (3 mantissa bits, ties to even), saturated to +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                      # a = m * 2^ex with m in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_EMIN)        # binade exponent, floored at the subnormal range
    step = np.ldexp(1.0, e - 3)
    q = np.minimum(np.round(a / step) * step, E4M3_MAX)
    return np.copysign(q, v)


# MXFP4 (the FP4 of the pages' FP8 x FP4 weights; OCP MX v1.0): E2M1 elements, values
# {0, 0.5, 1, 1.5, 2, 3, 4, 6}, with the same E8M0 scale per 32 elements
E2M1_MAX = 6.0
E2M1_EMAX = 2          # exponent of the largest E2M1 value (6 = 1.5 * 2^2)
E2M1_EMIN = 0          # exponent of the smallest normal (1.0); the subnormal is 0.5


def e2m1_round(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 value (1 mantissa bit, ties to even), saturated to +-6."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = np.maximum(ex - 1, E2M1_EMIN)
    step = np.ldexp(1.0, e - 1)
    q = np.minimum(np.round(a / step) * step, E2M1_MAX)
    return np.copysign(q, v)


def mx_block_exponent(amax: np.ndarray, emax: int = E4M3_EMAX) -> np.ndarray:
    """Shared block exponent floor(log2(amax)) - emax (8 for E4M3, 2 for E2M1), clamped to the E8M0
    range; -127 for amax = 0."""
    amax = np.asarray(amax, dtype=np.float64)
    _, ex = np.frexp(amax)
    se = (ex - 1) - emax
    se = np.clip(se, -127, 127)
    return np.where(amax > 0, se, -127).astype(np.int64)


def _qdq_last_axis(a: np.ndarray, fmt: str = "e4m3") -> np.ndarray:
    rnd, emax = (e4m3_round, E4M3_EMAX) if fmt == "e4m3" else (e2m1_round, E2M1_EMAX)
    n = a.shape[-1]
    nb = -(-n // MX_BLOCK)
    pad = nb * MX_BLOCK - n
    if pad:
        a = np.concatenate([a, np.zeros(a.shape[:-1] + (pad,))], axis=-1)
    b = a.reshape(a.shape[:-1] + (nb, MX_BLOCK))
    se = mx_block_exponent(np.abs(b).max(axis=-1), emax)[..., None]
    scale = np.ldexp(1.0, se)
    q = rnd(b / scale) * scale
    q = q.reshape(a.shape)
    return q[..., :n] if pad else q


def mx_qdq(a: np.ndarray, axis: int, fmt: str = "e4m3") -> np.ndarray:
    """Quantise to MXFP8 (fmt "e4m3") or MXFP4 ("e2m1") with 32-element blocks running along
    `axis`, then dequantise (fp64)."""
    a = np.moveaxis(np.asarray(a, dtype=np.float64), axis, -1)
    return np.moveaxis(_qdq_last_axis(a, fmt), -1, axis)


def mx_qdq_segments(a: np.ndarray, starts: np.ndarray) -> np.ndarray:
    """MXFP8 qdq along axis 0 with blocks restarting at each segment start (expert group).

    Rows [starts[i], starts[i+1]) form one segment; blocks of 32 rows run from the segment's
    first row and the last, shorter block is padded with zeros.
    """
    a = np.asarray(a, dtype=np.float64)
    out = np.empty_like(a)
    for i in range(len(starts) - 1):
        lo, hi = int(starts[i]), int(starts[i + 1])
        if hi > lo:
            out[lo:hi] = mx_qdq(a[lo:hi], axis=0)
    return out


# ----------------------------------------------------------------------------------------------
# forward
# ----------------------------------------------------------------------------------------------
def _as64(a):
    return np.asarray(a, dtype=np.float64)


def _stored_bf16(a):
    """a as the layer stores it between its forward and its backward: an fp32 value rounded to
    bf16 (to nearest, ties to even), read back exactly."""
    u = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = ((u + ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)) >> np.uint64(16)) << np.uint64(16)
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def forward(x, topk_idx, topk_w, W13, W2, *, mxfp8: bool = False, fp8_fp4: bool = False, keep: bool = False):
    """y[t] = sum_j w[t,j] * W2[e] (silu(W13[e,:I] x[t]) * (W13[e,I:] x[t])), e = topk_idx[t,j].

    Evaluated per expert group in sorted (routed) order.  With keep=True also returns the
    intermediates in sorted order: X_perm, g, u, h, o (and the routing dict).  fp8_fp4: the FP8 x
    FP4 forward the pages list for DeepGEMM's Mega MoE (wire.sakhanda.co, "Prime Intellect пусна
    Prime Mega MoE", section "Как се сравнява с други слети MoE опции?", data types row), read as MXFP8 activations (X, h) times
    MXFP4 weights (W13, W2), each blocked along its contraction.
    """
    if fp8_fp4:
        mxfp8 = True
    x, W13, W2 = _as64(x), _as64(W13), _as64(W2)
    T, H = x.shape
    E, I2, _ = W13.shape
    I = I2 // 2
    k = topk_idx.shape[1]
    r = route(topk_idx, E)
    wflat = _as64(topk_w).reshape(-1)
    X = permute_rows(x, r["perm"], k)
    if mxfp8:
        X = mx_qdq(X, axis=1)                # activations quantised along H (the contraction)
    S = T * k
    g = np.zeros((S, I)); u = np.zeros((S, I)); h = np.zeros((S, I)); o = np.zeros((S, H))
    for e in range(E):
        lo, hi = r["off"][e], r["off"][e + 1]
        if hi == lo:
            continue
        Wg, Wu, Wd = W13[e, :I], W13[e, I:], W2[e]
        if mxfp8:
            wf = "e2m1" if fp8_fp4 else "e4m3"
            Wg, Wu = mx_qdq(Wg, axis=1, fmt=wf), mx_qdq(Wu, axis=1, fmt=wf)
            Wd = mx_qdq(Wd, axis=1, fmt=wf)  # W2[e] is [H, I]: blocks along I, the contraction
        g[lo:hi] = X[lo:hi] @ Wg.T
        u[lo:hi] = X[lo:hi] @ Wu.T
        h[lo:hi] = silu(g[lo:hi]) * u[lo:hi]
        hq = mx_qdq(h[lo:hi], axis=1) if mxfp8 else h[lo:hi]
        o[lo:hi] = hq @ Wd.T
    w_sorted = wflat[r["perm"]]
    y = unpermute_sum(w_sorted[:, None] * o, r["inv"], T, k)
    if keep:
        return y, {"route": r, "X_perm": X, "g": g, "u": u, "h": h, "o": o, "w_sorted": w_sorted}
    return y


# ----------------------------------------------------------------------------------------------
# backward of the loss L = <dy, y>
# ----------------------------------------------------------------------------------------------
def backward(dy, x, topk_idx, topk_w, W13, W2, *, mxfp8: bool = False, fp8_bwd: bool = False, keep: bool = False):
    """Gradients of <dy, y> with respect to x, W13, W2 and topk_w.

    Per slot (t, j) routed to expert e, with g, u, h from the forward:
      dA = W2[e]^T dy[t]                    dtopk_w[t, j] = <dA, h>   (= <dy[t], o[t, j]>)
      dh = w * dA                           dg = dh * u * s(g) * (1 + g * (1 - s(g)))
      du = dh * silu(g)                     dx[t] += W13[e,:I]^T dg + W13[e,I:]^T du
      dW2[e] += dy[t] (w h)^T               dW13[e,:I] += dg x[t]^T,  dW13[e,I:] += du x[t]^T
    In MXFP8 mode each GEMM operand is quantised along that GEMM's contraction axis first
    (for the weight gradients the contraction runs over the tokens of one expert group); with
    fp8_bwd only the backward GEMMs' operands are, the forward (g, u, h) staying exact.  With a
    quantised backward, g and u enter it as the layer stores them, in bf16: the quantised codes of
    [dg|du] and w h are decided from those values.
    """
    dy, x, W13, W2 = _as64(dy), _as64(x), _as64(W13), _as64(W2)
    T, H = x.shape
    E, I2, _ = W13.shape
    I = I2 // 2
    k = topk_idx.shape[1]
    qb = mxfp8 or fp8_bwd                    # backward GEMM operands quantised
    _, fw = forward(x, topk_idx, topk_w, W13, W2, mxfp8=mxfp8, keep=True)
    r = fw["route"]
    off = r["off"]
    g, u, h, w_s = fw["g"], fw["u"], fw["h"], fw["w_sorted"]
    if qb:
        # the E4M3 codes of [dg|du] and w h are decided from the pre-activations as the layer
        # keeps them for its backward, in bf16; both sides decide from the same stored values
        g, u = _stored_bf16(g), _stored_bf16(u)
        h = silu(g) * u
    X = fw["X_perm"]                         # already quantised along H in MXFP8 mode
    X_raw = permute_rows(x, r["perm"], k)
    dY = permute_rows(dy, r["perm"], k)
    dYq = mx_qdq(dY, axis=1) if qb else dY
    S = T * k
    dA = np.zeros((S, I)); dG = np.zeros((S, 2 * I)); Hw = np.zeros((S, I)); dXp = np.zeros((S, H))
    dW13 = np.zeros_like(W13); dW2 = np.zeros_like(W2)
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        Wd = mx_qdq(W2[e], axis=0) if qb else W2[e]          # contraction over H: blocks along H
        dA[lo:hi] = dYq[lo:hi] @ Wd
        sg = sigmoid(g[lo:hi])
        dh = w_s[lo:hi, None] * dA[lo:hi]
        dG[lo:hi, :I] = dh * u[lo:hi] * sg * (1.0 + g[lo:hi] * (1.0 - sg))
        dG[lo:hi, I:] = dh * g[lo:hi] * sg
        Hw[lo:hi] = w_s[lo:hi, None] * h[lo:hi]
        W = mx_qdq(W13[e], axis=0) if qb else W13[e]        # contraction over 2I: blocks along 2I
        dGq = mx_qdq(dG[lo:hi], axis=1) if qb else dG[lo:hi]
        dXp[lo:hi] = dGq @ W
    dtw_sorted = np.einsum("si,si->s", dA, h)
    if qb:
        a6, b6 = mx_qdq_segments(dY, off), mx_qdq_segments(Hw, off)
        a7, b7 = mx_qdq_segments(dG, off), mx_qdq_segments(X_raw, off)
    else:
        a6, b6, a7, b7 = dY, Hw, dG, X_raw
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue                          # an expert without tokens has zero weight gradients
        dW2[e] = a6[lo:hi].T @ b6[lo:hi]
        dW13[e] = a7[lo:hi].T @ b7[lo:hi]
    dx = unpermute_sum(dXp, r["inv"], T, k)
    dtopk_w = np.empty(S)
    dtopk_w[r["perm"]] = dtw_sorted
    dtopk_w = dtopk_w.reshape(T, k)
    out = {"dx": dx, "dW13": dW13, "dW2": dW2, "dtopk_w": dtopk_w}
    if keep:
        out.update({"fwd": fw, "dY_perm": dY, "dA": dA, "dG": dG, "Hw": Hw, "dXpart": dXp})
    return out


# ----------------------------------------------------------------------------------------------
# sampled evaluation for full-size checks: a few tokens or a few experts at a time
# ----------------------------------------------------------------------------------------------
def forward_tokens(x, topk_idx, topk_w, W13, W2, tokens, *, mxfp8: bool = False, fp8_fp4: bool = False):
    """y[t] for the listed tokens only, one slot at a time (BF16 / MXFP8 / FP8 x FP4 as in `forward`)."""
    I = W13.shape[1] // 2
    wf = "e2m1" if fp8_fp4 else "e4m3"
    mxfp8 = mxfp8 or fp8_fp4
    out = np.zeros((len(tokens), x.shape[1]))
    for n, t in enumerate(tokens):
        xt = _as64(x[t])
        if mxfp8:
            xt = mx_qdq(xt[None], axis=1)[0]
        for j in range(topk_idx.shape[1]):
            e = int(topk_idx[t, j])
            W = _as64(W13[e]); Wd = _as64(W2[e])
            if mxfp8:
                W = mx_qdq(W, axis=1, fmt=wf); Wd = mx_qdq(Wd, axis=1, fmt=wf)
            g = W[:I] @ xt
            u = W[I:] @ xt
            hh = silu(g) * u
            if mxfp8:
                hh = mx_qdq(hh[None], axis=1)[0]
            out[n] += float(topk_w[t, j]) * (Wd @ hh)
    return out


def _row_qdq(v):
    return mx_qdq(v[None], axis=1)[0]


def backward_tokens(dy, x, topk_idx, topk_w, W13, W2, tokens, *, mxfp8: bool = False, fp8_bwd: bool = False):
    """dx[t] and dtopk_w[t, :] for the listed tokens only (fp64), with the quantisation points of
    `backward`: in MXFP8 mode x along H and W13 along H (forward); in MXFP8 and fp8_bwd modes dy
    along H, W13 along 2I and W2 along H (dgrad), [dg|du] along 2I."""
    I = W13.shape[1] // 2
    k = topk_idx.shape[1]
    qb = mxfp8 or fp8_bwd
    dx = np.zeros((len(tokens), x.shape[1]))
    dtw = np.zeros((len(tokens), k))
    for n, t in enumerate(tokens):
        xt, dyt = _as64(x[t]), _as64(dy[t])
        if mxfp8:
            xt = _row_qdq(xt)
        if qb:
            dyt = _row_qdq(dyt)
        for j in range(k):
            e = int(topk_idx[t, j])
            W = _as64(W13[e]); Wd = _as64(W2[e])
            Wf = mx_qdq(W, axis=1) if mxfp8 else W          # forward: contraction over H
            Wb = mx_qdq(W, axis=0) if qb else W             # dgrad: contraction over 2I
            Wdb = mx_qdq(Wd, axis=0) if qb else Wd          # dgrad: contraction over H
            g = Wf[:I] @ xt
            u = Wf[I:] @ xt
            if qb:
                g, u = _stored_bf16(g), _stored_bf16(u)
            sg = sigmoid(g)
            dA = Wdb.T @ dyt
            dtw[n, j] = dA @ (silu(g) * u)
            dh = float(topk_w[t, j]) * dA
            dG = np.concatenate([dh * u * sg * (1.0 + g * (1.0 - sg)), dh * g * sg])
            if qb:
                dG = _row_qdq(dG)
            dx[n] += Wb.T @ dG
    return dx, dtw


def wgrad_experts(dy, x, topk_idx, topk_w, W13, W2, experts, *, mxfp8: bool = False, fp8_bwd: bool = False):
    """(dW13[e], dW2[e]) for the listed experts only (fp64).  The forward (MXFP8 mode) and dgrad
    (MXFP8 and fp8_bwd modes) operands are quantised as in `backward`, and the weight-gradient
    operands along the expert's tokens in slot order (blocks of 32 from the group's first token,
    zero-padded tail)."""
    I = W13.shape[1] // 2
    k = topk_idx.shape[1]
    qb = mxfp8 or fp8_bwd
    flat = np.asarray(topk_idx).reshape(-1)
    wflat = _as64(topk_w).reshape(-1)
    res = []
    for e in experts:
        slots = np.nonzero(flat == e)[0]
        t = slots // k
        X = _as64(x[t]); dY = _as64(dy[t]); w = wflat[slots][:, None]
        W = _as64(W13[e]); Wd = _as64(W2[e])
        Xf, dYb, Wf, Wdb = X, dY, W, Wd
        if mxfp8:
            Xf, Wf = mx_qdq(X, axis=1), mx_qdq(W, axis=1)
        if qb:
            dYb, Wdb = mx_qdq(dY, axis=1), mx_qdq(Wd, axis=0)
        g = Xf @ Wf[:I].T
        u = Xf @ Wf[I:].T
        if qb:
            g, u = _stored_bf16(g), _stored_bf16(u)
        sg = sigmoid(g)
        h = g * sg * u
        dA = dYb @ Wdb
        dh = w * dA
        dG = np.concatenate([dh * u * sg * (1.0 + g * (1.0 - sg)), dh * g * sg], axis=1)
        Hw = w * h
        if qb and len(slots):
            seg = np.array([0, len(slots)])
            dY, Hw = mx_qdq_segments(dY, seg), mx_qdq_segments(Hw, seg)
            dG, X = mx_qdq_segments(dG, seg), mx_qdq_segments(X, seg)
        res.append((dG.T @ X, dY.T @ Hw))
    return res


# ----------------------------------------------------------------------------------------------
# router: the step before the layer (the pages' layer benchmark leaves it out: ic.work analysis,
# section "跑分背后的理想假设与闭源软肋"); each token's routing weights aggregate the expert
# outputs (kongchang.com, "为什么 MoE 训练特别需要融合内核").  Readings where the pages are silent:
# the k largest logits are selected, ties to the lower expert index, listed in descending order;
# the weights are the softmax over the selected logits (the full softmax renormalised over the
# top-k); the selection is piecewise constant, so the backward reaches only the selected logits.
# ----------------------------------------------------------------------------------------------
def router_forward(logits, k: int):
    """(topk_idx int32 [T, k], topk_w fp64 [T, k]) of router logits [T, E]."""
    L = _as64(logits)
    T, E = L.shape
    cols = np.broadcast_to(np.arange(E), L.shape)
    order = np.lexsort((cols, -L), axis=1)          # by logit descending, then index ascending
    idx = order[:, :k]
    sel = np.take_along_axis(L, idx, axis=1)
    z = np.exp(sel - sel[:, :1])                    # the first selected logit is the largest
    return idx.astype(np.int32), z / z.sum(axis=1, keepdims=True)


def router_backward(topk_idx, topk_w, dtopk_w, E: int):
    """dlogits [T, E] of sum_j dtopk_w[t, j] * topk_w[t, j]: through the softmax over the selected
    logits, dl_j = w_j (dw_j - sum_i w_i dw_i); zero for experts a token did not select."""
    w, dw = _as64(topk_w), _as64(dtopk_w)
    g = w * (dw - (w * dw).sum(axis=1, keepdims=True))
    dl = np.zeros((w.shape[0], E))
    np.put_along_axis(dl, np.asarray(topk_idx, dtype=np.int64), g, axis=1)
    return dl
