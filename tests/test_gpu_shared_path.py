"""The shared-expert path of the layer, on its own (both decode paths).

K3 shape (hidden 7168, two bf16 shared experts of intermediate 1536) with 16
routed experts whose E2M1 codes are all zero: code 0 is +0, so every routed
expert contributes exactly 0 whatever the routing, and with top-16 of 16 the
layer output is the shared experts' sum (plus the residual). In the full
layer that sum is ~1e-5 of the routed part, so this is where its parity is
visible. Batch sizes 1, 5 and 8 cover both the one- and two-column-group
forms of the shared down GEMV; 9, 100 and 200 the dense tcgen05 GEMMs that
take over above the decode range (ragged token tiles of 128, and for the
down GEMM two columns per token).

On a handle made for batches (exact planes) the dense GEMMs serve the shared
experts from 4 tokens on (checked at 1, 4, 8 and 100 tokens).

Bar: relative L2 <= 1e-5 against the oracle's double sum on the decode
path (T <= 8): the kernel's f16 form of each bf16 weight row (a power-of-two
row scale) is exact, products of f16 values are exact in fp32, and only fp32
accumulation rounding remains. Above the decode range the contractions
(K = 7168, then 3072) run on tcgen05, whose accumulation of the exact bf16
products follows the tensor core's own summation rather than sequential
fp32 adds; measured 1.9e-5, bar 5e-5. (The shared part is ~1e-5 of a
layer's output, so either bar sits far inside the layer tolerance.)
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import bits_to_f64, check_ids_weights, rel_l2, to_dev_bf16

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS[1]
E = 16


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


def _zero_routed(torch, flags=0):
    import mxfp4_routed_expert_top_gb300 as dfm
    m = dfm.MoE(WL.H, E, E, WL.I, WL.n_shared, WL.Is, max_tokens=200, flags=flags)
    router = synth.router(WL.seed, WL.wcfg, 0, E, WL.H)
    shared = [synth.shared(WL.seed, WL.wcfg, 0, s, WL.H, WL.Is) for s in range(WL.n_shared)]
    zeros = torch.zeros(E * m.span_bytes, dtype=torch.uint8, device="cuda")
    m.load_experts(0, router=router, shared=shared)
    m.load_experts(0, experts=zeros, expert_begin=0, expert_count=E, src_is_device=True)
    torch.cuda.synchronize()
    return m, router, shared


@pytest.fixture(scope="module")
def zero_routed(torch):
    m, router, shared = _zero_routed(torch)
    yield m, router, shared
    m.close()


@pytest.fixture(scope="module")
def zero_routed_planes(torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    m, router, shared = _zero_routed(torch, dfm.PLANES)
    yield m, router, shared
    m.close()


@pytest.mark.parametrize("T", [1, 4, 8, 100])
def test_shared_only_layer_planes_handle(zero_routed_planes, torch, T):
    _check_shared_only(zero_routed_planes, torch, T, bar=1e-5 if T < 4 else 5e-5)


@pytest.mark.parametrize("T", [1, 5, 8, 9, 100, 200])
def test_shared_only_layer(zero_routed, torch, T):
    _check_shared_only(zero_routed, torch, T, bar=1e-5 if T <= 8 else 5e-5)


def _check_shared_only(handle, torch, T, bar):
    m, router, shared = handle
    x = np.stack([synth.token(WL.seed, 2, 4000 + t, WL.H) for t in range(T)])
    res = np.stack([synth.token(WL.seed, 2, 4100 + t, WL.H) for t in range(T)])
    out = torch.empty((T, WL.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, WL.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, E), dtype=torch.int32, device="cuda")
    w = torch.empty((T, E), dtype=torch.float32, device="cuda")
    m.forward(to_dev_bf16(x), T, out, ids, w, residual=to_dev_bf16(res), out_f32=out32)
    m.sync()
    got = out32.cpu().double().numpy() - bits_to_f64(res)
    for t in range(T):
        ref = sum(orc.shared_ffn(*s, bits_to_f64(x[t])) for s in shared)
        assert rel_l2(got[t], ref) <= bar, "token %d" % t
    # routing over all 16 experts: the set is all of them, weights a softmax
    rid, rw = orc.topk_softmax(orc.router_logits(router, x), E)
    check_ids_weights(ids.cpu().numpy(), w.cpu().double().numpy(), rid, rw)
