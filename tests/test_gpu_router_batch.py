"""Router logits of batches (more than 8 tokens) against the oracle.

The router is an fp32 linear map over the experts (Deltafin analysis, §5.1).
For batches the library holds the fp32 weights as three bf16 parts (high,
middle, low; their sum is the weight) and runs a bf16 GEMM on the tensor
cores with fp32 accumulation: every product is exact, so the logits carry
fp32 accumulation error only. Pins that hold whatever the order of the sums:
  * one-hot tokens (one column set to a power of two): each logit is a single
    weight times that power, so it must come back bit-exact. The synthetic
    weights are random fp32 values with all 24 significant bits set, so a
    dropped or mis-rounded part, or a part multiplied by the wrong column of
    x, changes the result;
  * Gaussian tokens: |logit - oracle| <= 1e-5 sum_j |x_j w_ej| at the K3
    shape (896 experts, hidden 7168) and at a ragged shape (200 experts: the
    second 128-row tile is part empty; token counts not multiples of 128),
    and the selection on those logits is the oracle's where the gap rule
    holds.
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import bits_to_f64, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _handle(H, E, max_tokens, seed, k=4, flags=0):
    """A handle whose layer 0 has only its router loaded (the router and
    top-k steps need nothing else)."""
    import mxfp4_routed_expert_top_gb300 as dfm
    m = dfm.MoE(H, E, k, 128, 1, 64, n_layers=1, max_tokens=max_tokens, flags=flags)
    router = synth.router(seed, 0, 0, E, H)
    m.load_experts(0, router=router)
    m.sync()
    return m, router


def _logits(torch, m, x_dev, T, E):
    out = torch.empty((T, E), dtype=torch.float32, device="cuda")
    m.step_router(0, x_dev, T, out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _bound(router, x):
    return 1e-5 * (np.abs(bits_to_f64(x)) @ np.abs(router.astype(np.float64)).T) + 1e-30


def _bf16_bits(v):
    return (np.asarray(v, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("T", [9, 130, 300])
def test_one_hot_tokens_exact(torch, T):
    H, E = 256, 200
    m, router = _handle(H, E, 300, seed=71)
    try:
        cols = (np.arange(T) * 37) % H
        scale = np.ldexp(1.0, (np.arange(T) % 5) - 2) * np.where(np.arange(T) % 2, -1.0, 1.0)
        x = np.zeros((T, H), dtype=np.uint16)
        x[np.arange(T), cols] = _bf16_bits(scale)
        got = _logits(torch, m, to_dev_bf16(x), T, E)
        want = (router[:, cols].T * scale[:, None].astype(np.float32)).astype(np.float32)
        # nearly every weight needs all three parts (the low 8 of its 24
        # significant bits are not all zero)
        assert np.mean((router.view(np.uint32) & 0xFF) > 0) > 0.99
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    finally:
        m.close()


@pytest.mark.parametrize("T", [4, 8])
def test_planes_handle_small_batches(torch, T):
    """Block-scaled handles take batches of 4-8 tokens through the tensor-core
    router too (one-hot tokens: bit-exact; Gaussian: the 1e-5 bound)."""
    import mxfp4_routed_expert_top_gb300 as dfm
    H, E = 256, 200
    m, router = _handle(H, E, 8, seed=73, flags=dfm.PLANES)
    try:
        cols = (np.arange(T) * 53) % H
        x = np.zeros((T, H), dtype=np.uint16)
        x[np.arange(T), cols] = _bf16_bits(np.ones(T))
        got = _logits(torch, m, to_dev_bf16(x), T, E)
        assert np.array_equal(got.view(np.uint32), router[:, cols].T.copy().view(np.uint32))
        x = np.stack([synth.token(73, 0, 60 + t, H) for t in range(T)])
        got = _logits(torch, m, to_dev_bf16(x), T, E)
        assert np.all(np.abs(got - orc.router_logits(router, x)) <= _bound(router, x))
    finally:
        m.close()


@pytest.mark.parametrize("T", [9, 130, 300])
def test_ragged_shape_gaussian(torch, T):
    H, E = 256, 200
    m, router = _handle(H, E, 300, seed=72)
    try:
        x = np.stack([synth.token(72, 0, 40 + t, H) for t in range(T)])
        got = _logits(torch, m, to_dev_bf16(x), T, E)
        ref = orc.router_logits(router, x)
        assert np.all(np.abs(got - ref) <= _bound(router, x))
    finally:
        m.close()


@pytest.fixture(scope="module")
def k3(torch):
    wl = synth.WORKLOADS[3]
    m, router = _handle(wl.H, wl.E, 512, seed=wl.seed, k=wl.k)
    yield wl, m, router
    m.close()


@pytest.mark.parametrize("T", [9, 64, 512])
def test_k3_shape(k3, torch, T):
    wl, m, router = k3
    x = np.stack([synth.token(wl.seed, wl.cfg_id, 3000 + t, wl.H) for t in range(T)])
    got = _logits(torch, m, to_dev_bf16(x), T, wl.E)
    ref = orc.router_logits(router, x)
    assert np.all(np.abs(got - ref) <= _bound(router, x))
    # the selection on these logits is the oracle's where the gap rule holds
    ids = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    m.step_topk(torch.from_numpy(got).cuda(), T, ids, w)
    torch.cuda.synchronize()
    rid, _ = orc.topk_softmax(ref, wl.k)
    srt = np.sort(ref, axis=1)[:, ::-1]
    ok = srt[:, wl.k - 1] - srt[:, wl.k] >= 1e-3
    assert ok.sum() > T // 2
    assert np.array_equal(ids.cpu().numpy()[ok], rid[ok])
