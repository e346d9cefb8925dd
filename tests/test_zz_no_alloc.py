"""The allocation-free routing entry point, moe_route_static, against the routing moe_fwd leaves in
its scratch buffer and against the oracle's routing.

moe_route_static is for callers that cannot allocate device memory (allocator hooks, runtimes
that reserve all memory up front, loops where an allocation would synchronise the device): its
working memory is a static device array inside the library.  Routing is integer work, so the
outputs must match bit for bit.  Two calls in a row check that what the shared array keeps from
the previous call does not leak into the next.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_permute_gb300 import inputs as gen

from _layer import DeviceLayer

pytestmark = pytest.mark.gpu

CASES = [
    gen.custom_config("noalloc_a", T=4096, H=256, I=128, E=128, k=8, seed=41),
    gen.custom_config("noalloc_b", T=3000, H=256, I=128, E=64, k=6, routing="zipf", seed=42),
]


def test_static_routing_matches_moe_fwd_twice_in_a_row(cuda_lib):
    bd = cuda_lib
    for cfg in CASES:
        inp = gen.make_inputs(cfg)
        L = DeviceLayer(bd, inp)
        L.fwd()                                    # the existing entry point, with its scratch
        S, E = cfg.S, cfg.E
        ref = {"counts": L.view(bd.MOE_VIEW_COUNTS, torch.int32, (E,)).clone(),
               "offsets": L.view(bd.MOE_VIEW_OFFSETS, torch.int32, (E + 1,)).clone(),
               "perm": L.view(bd.MOE_VIEW_PERM, torch.int32, (S,)).clone(),
               "inv": L.view(bd.MOE_VIEW_INV, torch.int32, (S,)).clone()}
        out = {"counts": torch.full((E,), -7, dtype=torch.int32, device="cuda"),
               "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
               "perm": torch.full((S,), -7, dtype=torch.int32, device="cuda"),
               "inv": torch.full((S,), -7, dtype=torch.int32, device="cuda")}
        bd.moe_route_static(L.idx, E, out["counts"], out["offsets"], out["perm"], out["inv"])
        torch.cuda.synchronize()
        for name in ref:
            assert torch.equal(out[name], ref[name]), (cfg.name, name)
        assert int(out["offsets"][-1]) == S
        assert np.array_equal(np.sort(out["perm"].cpu().numpy()), np.arange(S))
        r = oracle.route(inp.topk_idx, E)
        for name, key in (("counts", "cnt"), ("offsets", "off"), ("perm", "perm"), ("inv", "inv")):
            assert np.array_equal(out[name].cpu().numpy(), r[key]), (cfg.name, name)


def _static_route(bd, idx_np, E):
    S = idx_np.size
    idx = torch.from_numpy(np.ascontiguousarray(idx_np)).cuda()
    out = {"counts": torch.full((E,), -7, dtype=torch.int32, device="cuda"),
           "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
           "perm": torch.full((S,), -7, dtype=torch.int32, device="cuda"),
           "inv": torch.full((S,), -7, dtype=torch.int32, device="cuda")}
    bd.moe_route_static(idx, E, out["counts"], out["offsets"], out["perm"], out["inv"])
    torch.cuda.synchronize()
    return {n: t.cpu().numpy() for n, t in out.items()}


def test_static_routing_drops_out_of_range_ids(cuda_lib):
    """Slots whose expert id lies outside [0, E) are dropped: inv = -1 for them, and the sorted
    positions they leave free at the end of perm hold -1; the valid slots route as the oracle routes
    them alone."""
    bd = cuda_lib
    E, k = 16, 4
    rng = np.random.default_rng(7)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(700)]).astype(np.int32)
    bad = [(3, 1, -1), (10, 0, E), (10, 3, E + 5), (699, 2, -100)]
    for t, j, v in bad:
        idx[t, j] = v
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    slots = np.nonzero(valid)[0]
    r = oracle.route(flat[valid], E)            # the valid slots, in slot order
    want_perm = np.full(flat.size, -1, dtype=np.int64)
    want_perm[:slots.size] = slots[r["perm"]]
    want_inv = np.full(flat.size, -1, dtype=np.int64)
    want_inv[slots] = r["inv"]
    for _ in range(2):                          # twice: nothing of the first call leaks into the second
        got = _static_route(bd, idx, E)
        assert np.array_equal(got["counts"], r["cnt"])
        assert np.array_equal(got["offsets"], r["off"]) and got["offsets"][-1] == flat.size - len(bad)
        assert np.array_equal(got["perm"], want_perm)
        assert np.array_equal(got["inv"], want_inv)


def test_static_routing_rejects_sizes_beyond_its_array(cuda_lib):
    bd = cuda_lib
    T, k, E = 300000, 8, 128          # 2 * ceil(2.4M / 2048) * 128 > 65536
    idx = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    rc = bd.LIB.moe_route_static(idx.data_ptr(), T, k, E, idx.data_ptr(), idx.data_ptr(), idx.data_ptr(),
                                 idx.data_ptr(), None)
    assert rc == bd.ERR["MOE_ERR_UNSUPPORTED"]
    assert bd.LIB.moe_route_static(idx.data_ptr(), 4, 9, 8, idx.data_ptr(), idx.data_ptr(), idx.data_ptr(),
                                   idx.data_ptr(), None) == bd.ERR["MOE_ERR_SHAPE"]
