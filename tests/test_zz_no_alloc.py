"""The allocation-free routing entry point (df_moe_route_noalloc).

Some callers cannot allocate device memory: an engine that has already split
all of HBM among its own pools, or a decode loop that must not take the
device-wide synchronisation an allocation can cause. For them the library
routes tokens with its scratch in a fixed static device array. This file runs
last (pytest collects it last) so that a failure here leaves every other
result in place; it also passes on its own in a fresh process.

Two calls in a row are compared with the handle-based entry points
(df_moe_step_router + df_moe_step_topk) on the same inputs: ids exactly,
routing weights within 1e-5, the tolerance the other tests use.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def test_route_noalloc_matches_handle_path(torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    wl = synth.WORKLOADS[1]
    E, H, k = wl.E, wl.H, wl.k
    router = synth.router(wl.seed, wl.wcfg, 0, E, H)
    router_dev = torch.from_numpy(router).cuda()
    # a handle with the same router, for the existing entry points
    with dfm.MoE(H, E, k, 64, 0, 0, max_tokens=8) as m:
        m.load_experts(0, router=router)
        for call, T in enumerate((8, 3)):   # two calls in a row
            x = np.stack([synth.token(wl.seed, wl.cfg_id, 40000 + 10 * call + t, H)
                          for t in range(T)])
            xd = torch.from_numpy(x.view(np.int16)).cuda()
            ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
            w = torch.empty((T, k), dtype=torch.float32, device="cuda")
            dfm.route_noalloc(router_dev, E, H, xd, T, k, ids, w)
            logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
            ids_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
            w_ref = torch.empty((T, k), dtype=torch.float32, device="cuda")
            m.step_router(0, xd, T, logits)
            m.step_topk(logits, T, ids_ref, w_ref)
            torch.cuda.synchronize()
            assert np.array_equal(ids.cpu().numpy(), ids_ref.cpu().numpy())
            assert np.max(np.abs(w.cpu().numpy() - w_ref.cpu().numpy())) <= 1e-5


def test_route_noalloc_rejects_oversized_calls(torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    E, H, k, T = 896, 7168, 16, 98    # needs 4 * 98 * 896 > 262,144 floats
    router = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(dfm.DfMoeError) as ei:
        dfm.route_noalloc(router, E, H, x, T, k, ids, w)
    assert ei.value.code == -5
    assert "scratch" in str(ei.value)
