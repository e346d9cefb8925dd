"""Seeded synthetic inputs for the MoE expert layer.

This module is shared by the tests, `bench.py` and the smoke check. It draws random numbers and
rounds them to bf16; it holds none of the layer's arithmetic (no routing bookkeeping, no GEMM,
no activation). The top-k expert ids and their weights stand in for a router, which the pages
leave out of their single-layer benchmark ("random routing, router cost excluded": ic.work
analysis, section "跑分背后的理想假设与闭源软肋"; MarkTechPost, "How fast is Prime Mega MoE?").

Recipe (every array from numpy PCG64; a tensor is drawn in chunks of 2^24 elements, chunk c of
tensor stream id i from its own generator keyed by `(seed, i, c)`, so that chunks can be drawn
in parallel and the result does not depend on the number of threads):

* x, dy ~ N(0, 1); W13 [E, 2I, H] ~ N(0, std = 1/sqrt(H)); W2 [E, H, I] ~ N(0, std = 1/sqrt(I)).
  All are drawn in float32 and rounded to bf16 (round to nearest, ties to even).
* uniform routing: each token takes the first k entries of its own random permutation of the E
  experts (k distinct experts, uniformly).
* zipf routing: expert popularity p_r proportional to r^-s (s = 1.2) over ranks r = 1..E, with the
  `zero_experts` lowest-ranked experts given popularity 0; ranks are mapped to experts by a random
  permutation; each token draws k distinct experts without replacement weighted by popularity
  (Gumbel-top-k on log p).
* top-k weights: softmax over k N(0, 1) logits (one per chosen expert), computed in float64 and
  stored as float32.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

# stream ids of the per-tensor generators
_S_ROUTE, _S_LOGIT, _S_X, _S_W13, _S_W2, _S_DY, _S_PERM, _S_RLOGIT, _S_DTW = range(9)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    precision: str = "bf16"          # "bf16", "mxfp8", "fp8_bwd" (BF16 forward, MXFP8 backward) or
                                     # "fp8_fp4" (forward only: MXFP8 activations x MXFP4 weights)
    routing: str = "uniform"         # "uniform" or "zipf"
    seed: int = 1000
    zipf_s: float = 1.2
    zero_experts: int = 4

    @property
    def S(self) -> int:
        return self.T * self.k

    def fwd_flops(self) -> float:
        """Algorithmic forward FLOPs 2*T*k*H*3I (two expert linears, gate+up then down)."""
        return 2.0 * self.T * self.k * self.H * 3 * self.I


# The five workloads: a tiny layer, the Qwen3-30B-A3B- and Qwen3-235B-A22B-shaped layers the pages
# benchmark (128 experts, top-8, 16,384 tokens), and a Zipf-skewed routing stress on the 30B shape.
CONFIGS = {
    "tiny": LayerConfig("tiny", T=256, H=256, I=128, E=8, k=2, seed=1000),
    "qwen3_30b_a3b": LayerConfig("qwen3_30b_a3b", T=16384, H=2048, I=768, E=128, k=8, seed=1001),
    "qwen3_30b_a3b_mxfp8": LayerConfig("qwen3_30b_a3b_mxfp8", T=16384, H=2048, I=768, E=128, k=8,
                                       precision="mxfp8", seed=1001),
    "qwen3_30b_a3b_fp8_bwd": LayerConfig("qwen3_30b_a3b_fp8_bwd", T=16384, H=2048, I=768, E=128, k=8,
                                         precision="fp8_bwd", seed=1001),
    "qwen3_30b_a3b_fp8_fp4": LayerConfig("qwen3_30b_a3b_fp8_fp4", T=16384, H=2048, I=768, E=128, k=8,
                                         precision="fp8_fp4", seed=1001),
    "qwen3_235b_a22b": LayerConfig("qwen3_235b_a22b", T=16384, H=4096, I=1536, E=128, k=8, seed=1003),
    "qwen3_235b_a22b_mxfp8": LayerConfig("qwen3_235b_a22b_mxfp8", T=16384, H=4096, I=1536, E=128, k=8,
                                         precision="mxfp8", seed=1003),
    "skew_zipf_16k": LayerConfig("skew_zipf_16k", T=16384, H=2048, I=768, E=128, k=8,
                                 routing="zipf", seed=1004),
    "skew_zipf_4k": LayerConfig("skew_zipf_4k", T=4096, H=2048, I=768, E=128, k=8,
                                routing="zipf", seed=1004),
    # the 30B layer shape at a quarter of the tokens: inputs still larger than L2, a few GB on the
    # device, small enough for a many-pass profiler capture
    "profile_30b_t4096": LayerConfig("profile_30b_t4096", T=4096, H=2048, I=768, E=128, k=8, seed=1001),
    # the 30B layer's per-expert work (about 1024 routed rows per expert) on 32 experts: the
    # GEMMs' arithmetic intensity of the full workload at a quarter of its device footprint
    "profile_30b_e32": LayerConfig("profile_30b_e32", T=4096, H=2048, I=768, E=32, k=8, seed=1001),
    "profile_30b_e32_mxfp8": LayerConfig("profile_30b_e32_mxfp8", T=4096, H=2048, I=768, E=32, k=8,
                                         precision="mxfp8", seed=1001),
    "profile_30b_e32_fp8_fp4": LayerConfig("profile_30b_e32_fp8_fp4", T=4096, H=2048, I=768, E=32, k=8,
                                           precision="fp8_fp4", seed=1001),
}


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    r += np.uint32(0x7FFF)
    r += u
    r >>= np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_CHUNK = 1 << 24


def _normal_bf16(seed: int, stream: int, shape, std: float) -> np.ndarray:
    """N(0, std^2) rounded to bf16, chunk c from the generator keyed (seed, stream, c)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)

    def fill(c: int) -> None:
        s0 = c * _CHUNK
        m = min(_CHUNK, n - s0)
        v = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, c]))).standard_normal(
            m, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s0:s0 + m] = f32_to_bf16_bits(v)

    chunks = (n + _CHUNK - 1) // _CHUNK
    workers = min(chunks, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else 1)
    if workers <= 1:
        for c in range(chunks):
            fill(c)
    else:
        with _cf.ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(fill, range(chunks)))
    return out.reshape(shape)


def routing(cfg: LayerConfig) -> tuple[np.ndarray, np.ndarray]:
    """(topk_idx int32 [T, k], topk_w float32 [T, k]) for the configuration's routing recipe."""
    T, E, k = cfg.T, cfg.E, cfg.k
    if k > E:
        raise ValueError("k > E")
    rng = _rng(cfg.seed, _S_ROUTE)
    if cfg.routing == "uniform":
        keys = rng.random((T, E))
    elif cfg.routing == "zipf":
        if E - cfg.zero_experts < k:
            raise ValueError("too few experts with non-zero popularity for top-k")
        ranks = np.arange(1, E + 1, dtype=np.float64)
        pop = ranks ** (-cfg.zipf_s)
        pop[E - cfg.zero_experts:] = 0.0
        pop /= pop.sum()
        expert_of_rank = _rng(cfg.seed, _S_PERM).permutation(E)
        p = np.empty(E)
        p[expert_of_rank] = pop
        with np.errstate(divide="ignore"):
            logp = np.log(p)
        gumbel = -np.log(-np.log(rng.random((T, E))))
        keys = -(logp[None, :] + gumbel)        # ascending sort of keys = descending score
    else:
        raise ValueError(cfg.routing)
    idx = np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    logits = _rng(cfg.seed, _S_LOGIT).standard_normal((T, k))
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return np.ascontiguousarray(idx), np.ascontiguousarray(w)


@dataclasses.dataclass
class LayerInputs:
    """bf16 tensors are held as uint16 bit patterns; `f32(name)` widens them exactly."""
    cfg: LayerConfig
    x: np.ndarray          # uint16 [T, H]
    topk_idx: np.ndarray   # int32 [T, k]
    topk_w: np.ndarray     # float32 [T, k]
    W13: np.ndarray        # uint16 [E, 2I, H]  (rows [0, I) gate, [I, 2I) up)
    W2: np.ndarray         # uint16 [E, H, I]
    dy: np.ndarray         # uint16 [T, H]

    def f32(self, name: str) -> np.ndarray:
        return bf16_bits_to_f32(getattr(self, name))

    def f64(self, name: str) -> np.ndarray:
        a = getattr(self, name)
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def make_inputs(cfg: LayerConfig | str, *, with_weights: bool = True, with_dy: bool = True) -> LayerInputs:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    T, H, I, E = cfg.T, cfg.H, cfg.I, cfg.E
    idx, w = routing(cfg)
    x = _normal_bf16(cfg.seed, _S_X, (T, H), 1.0)
    W13 = _normal_bf16(cfg.seed, _S_W13, (E, 2 * I, H), 1.0 / np.sqrt(H)) if with_weights else None
    W2 = _normal_bf16(cfg.seed, _S_W2, (E, H, I), 1.0 / np.sqrt(I)) if with_weights else None
    dy = _normal_bf16(cfg.seed, _S_DY, (T, H), 1.0) if with_dy else None
    return LayerInputs(cfg, x, idx, w, W13, W2, dy)


def router_inputs(cfg: LayerConfig | str, *, tie_step: float = 0.0) -> tuple[np.ndarray, np.ndarray]:
    """(router logits float32 [T, E] ~ N(0, 1), upstream gradient of the top-k weights float32
    [T, k] ~ N(0, 1)) for the router that precedes the layer.  tie_step > 0 rounds the logits to
    multiples of it, so that tokens carry equal logits (ties)."""
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    logits = _rng(cfg.seed, _S_RLOGIT).standard_normal((cfg.T, cfg.E), dtype=np.float32)
    if tie_step > 0:
        logits = (np.round(logits / np.float32(tie_step)) * np.float32(tie_step)).astype(np.float32)
    dtw = _rng(cfg.seed, _S_DTW).standard_normal((cfg.T, cfg.k), dtype=np.float32)
    return np.ascontiguousarray(logits), np.ascontiguousarray(dtw)


def custom_config(name="custom", **kw) -> LayerConfig:
    return LayerConfig(name, **kw)
