"""The grouped GEMMs' bounded pipeline waits, run out on purpose.

Every wait in the GEMM pipelines gives up after a limit and the kernel records MOE_DEV_TIMEOUT,
drains what it has in flight, frees its tensor memory and returns; it never traps or hangs (the
pages' lesson from a persistent kernel that deadlocked: ic.work analysis, section
"算子下沉时代的硬件死锁暗礁").  Here the producer warps are told to issue no operand loads, so the
MMA warps wait for stages that never fill, with no copy in flight, and the limit is short.  The
same scratch must then serve a normal layer that matches the oracle."""
import time

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer, f64, rel_fro

pytestmark = pytest.mark.gpu

LIMIT = 200_000          # SM cycles: about 0.1 ms at 2 GHz


def test_withheld_loads_time_out_then_the_scratch_works_again(cuda_lib):
    bd = cuda_lib
    inp = gen.make_inputs("tiny")
    L = DeviceLayer(bd, inp)
    L.scratch.set_wait_limit(LIMIT, bd.MOE_TEST_WITHHOLD_LOADS)
    t0 = time.time()
    L.fwd(flags=bd.MOE_FLAG_SAVE_GU)           # single-CTA GEMMs
    torch.cuda.synchronize()
    assert L.status() == bd.MOE_DEV_TIMEOUT
    L.bwd()                                    # also the two-SM (cluster) GEMMs
    torch.cuda.synchronize()
    assert L.status() == bd.MOE_DEV_TIMEOUT
    assert time.time() - t0 < 60               # every wait is bounded
    assert L.status() == bd.MOE_DEV_OK         # reading cleared the word

    L.scratch.set_wait_limit(0, 0)             # the default limit, loads issued
    L.fwd(flags=bd.MOE_FLAG_SAVE_GU)
    L.bwd(flags=bd.MOE_FLAG_REUSE_FWD)
    torch.cuda.synchronize()
    assert L.status() == bd.MOE_DEV_OK
    args = (inp.f64("x"), inp.topk_idx, inp.f64("topk_w"), inp.f64("W13"), inp.f64("W2"))
    g = oracle.backward(inp.f64("dy"), *args)
    assert rel_fro(f64(L.y), oracle.forward(*args)) < 1e-2
    for name, got in (("dx", L.dx), ("dW13", L.dW13), ("dW2", L.dW2), ("dtopk_w", L.dtw)):
        assert rel_fro(f64(got), g[name]) < 1e-2, name
    assert np.isfinite(f64(L.y)).all()
