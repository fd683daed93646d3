"""The allocation-free routing entry point (df_moe_route_noalloc).

Some callers cannot allocate device memory: an engine that has already split
all of HBM among its own pools, or a decode loop that must not take the
device-wide synchronisation an allocation can cause. For them the library
routes tokens with its scratch in a fixed static device array. This file runs
last (pytest collects it last) so that a failure here leaves every other
result in place; it also passes on its own in a fresh process.

Calls in a row (T = 8, 3, 1 and 73, the largest T whose scratch fits at K3
shape; T = 1 launches the one-token router without the in-router top-k, a
launch the handle path never makes) are compared with the handle-based entry
points (df_moe_step_router + df_moe_step_topk) on the same inputs, and with
the oracle on tokens drawn with the routing-gap rule: ids exactly, routing
weights within 1e-5, the tolerance the other tests use.
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


def _gap_tokens(router, wl, T, first_id):
    """T tokens whose k-th and (k+1)-th oracle logits differ by >= 1e-3."""
    import oracle as orc
    from moe_setup import gap_ok
    out = []
    for t in range(T):
        for r in range(synth.gen.REDRAWS_PER_TOKEN):
            x = synth.token(wl.seed, wl.cfg_id, first_id + t, wl.H, redraw=r)
            if gap_ok(orc.router_logits(router, x), wl.k):
                out.append(x)
                break
        else:
            raise RuntimeError("no token passed the gap rule")
    return np.stack(out)


def test_route_noalloc_matches_handle_path_and_oracle(torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    import oracle as orc
    from moe_setup import check_ids_weights
    wl = synth.WORKLOADS[1]
    E, H, k = wl.E, wl.H, wl.k
    router = synth.router(wl.seed, wl.wcfg, 0, E, H)
    router_dev = torch.from_numpy(router).cuda()
    # a handle with the same router, for the existing entry points
    with dfm.MoE(H, E, k, 64, 0, 0, max_tokens=73) as m:
        m.load_experts(0, router=router)
        for call, T in enumerate((8, 3, 1, 73)):   # calls in a row
            x = _gap_tokens(router, wl, T, 40000 + 100 * call)
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
            got_ids, got_w = ids.cpu().numpy(), w.cpu().numpy()
            # above 8 tokens the handle's router is a tiled GEMM that sums in
            # another order, so two selected logits closer than its rounding
            # may swap places: ids as sets, weights keyed by id
            check_ids_weights(got_ids, got_w, ids_ref.cpu().numpy(), w_ref.cpu().numpy())
            o_ids, o_w = orc.topk_softmax(orc.router_logits(router, x), k)
            check_ids_weights(got_ids, got_w, o_ids, o_w)


def test_route_noalloc_rejects_misaligned_router(torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    E, H, k, T = 8, 256, 2, 1
    buf = torch.zeros(E * H + 1, dtype=torch.float32, device="cuda")
    router = buf[1:].view(E, H)     # 4 bytes past a 16-byte boundary
    x = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(dfm.DfMoeError) as ei:
        dfm.route_noalloc(router, E, H, x, T, k, ids, w)
    assert ei.value.code == -1
    assert "router" in str(ei.value)


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
