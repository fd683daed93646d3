"""GPU parity of the routed experts above the decode range (T > 8): the
grouped tcgen05 GEMMs (default) and the register-fragment kernels they
replace (PREFILL_MMA_SYNC), through the C ABI against the oracle.

Tiny workload shape with a wider intermediate (H=256, I=128, 8 experts,
top-2; the GEMMs take K in chunks of 128 columns) so that the oracle can
check every assignment: with 512 tokens each expert holds ~128 of them,
several token blocks of both GEMMs (32 tokens of gate/up, 16 tokens of
down), and a ragged last block. A hot expert that every token picks covers
the largest item a batch can make.

Step bar: relative L2 <= 1e-5 per row. The GEMMs multiply f16 operands:
the weights as E2M1 values times 2^(e - r), r a per-row reference exponent
(exact within 26 octaves of the row's largest block), x exactly (f16 with a
power of two per token), and the down input h as a high and a low f16 part
(|h - hi - lo| <= 2^-22 |h|); accumulation is fp32.
"""
import dataclasses

import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import (Setup, bits_to_f64, check_ids_weights, check_out,
                       draw_tokens, rel_l2, to_dev_bf16)

pytestmark = pytest.mark.gpu

WL = dataclasses.replace(synth.WORKLOADS[0], I=128, name="tiny-h256-i128-e8-top2")


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module", params=["tcgen05", "mma_sync"])
def tiny(torch, request):
    s = Setup(WL, max_tokens=512, mma_sync_prefill=request.param == "mma_sync")
    s.path = request.param
    yield s
    s.close()


def _tokens(tiny, T, first_id):
    # routing ties do not matter for the expert steps (ids are inputs there)
    return np.stack([synth.token(WL.seed, WL.cfg_id, first_id + t, WL.H) for t in range(T)])


def _route(tiny, x):
    return orc.topk_softmax(orc.router_logits(tiny.routers[0], x), WL.k)


def _hot_ids(T, hot=3):
    """Every token's first choice is expert `hot`; the second cycles over
    the others."""
    ids = np.empty((T, WL.k), dtype=np.int32)
    others = [e for e in range(WL.E) if e != hot]
    for t in range(T):
        ids[t, 0] = hot
        ids[t, 1] = others[t % len(others)]
    return ids


def _check_gateup(tiny, torch, x, ids):
    T = x.shape[0]
    hbuf = torch.empty((T * WL.k, WL.I), dtype=torch.float32, device="cuda")
    tiny.m.step_expert_gateup(0, to_dev_bf16(x), T, torch.from_numpy(ids).cuda(), hbuf)
    torch.cuda.synchronize()
    got = hbuf.cpu().double().numpy()
    for t in range(T):
        xt = bits_to_f64(x[t])
        for j in range(WL.k):
            ref = orc.expert_gateup(tiny._span(0, ids[t, j]), WL.H, WL.I, xt)
            assert rel_l2(got[t * WL.k + j], ref) <= 1e-5, "token %d slot %d" % (t, j)
    return got


def _check_down(tiny, torch, ids, w, h):
    T = ids.shape[0]
    y = torch.empty((T, WL.H), dtype=torch.float32, device="cuda")
    tiny.m.step_expert_down(0, torch.from_numpy(h.astype(np.float32)).cuda(), T,
                            torch.from_numpy(ids).cuda(),
                            torch.from_numpy(w.astype(np.float32)).cuda(), y)
    torch.cuda.synchronize()
    got = y.cpu().double().numpy()
    h32 = h.astype(np.float32).astype(np.float64)
    for t in range(T):
        ref = sum(np.float64(np.float32(w[t, j])) *
                  orc.expert_down(tiny._span(0, ids[t, j]), WL.H, WL.I, h32[t * WL.k + j])
                  for j in range(WL.k))
        assert rel_l2(got[t], ref) <= 1e-5, "token %d" % t


@pytest.mark.parametrize("T", [9, 64, 300])
def test_gateup_step_batches(tiny, torch, T):
    x = _tokens(tiny, T, 7000 + T)
    ids, _ = _route(tiny, x)
    _check_gateup(tiny, torch, x, ids)


@pytest.mark.parametrize("T", [9, 300])
def test_down_step_batches(tiny, torch, T):
    x = _tokens(tiny, T, 8000 + T)
    ids, w = _route(tiny, x)
    h = np.stack([orc.expert_gateup(tiny._span(0, ids[t, j]), WL.H, WL.I, bits_to_f64(x[t]))
                  for t in range(T) for j in range(WL.k)])
    _check_down(tiny, torch, ids, w, h)


def test_hot_expert_steps(tiny, torch):
    # 512 tokens on one expert: 16 gate/up token blocks, 32 down token blocks
    T = 512
    x = _tokens(tiny, T, 9000)
    ids = _hot_ids(T)
    h = _check_gateup(tiny, torch, x, ids)
    w = np.full((T, WL.k), 0.5)
    _check_down(tiny, torch, ids, w, h)


@pytest.mark.parametrize("T", [9, 33, 512])
def test_forward_batches(tiny, torch, T):
    x = draw_tokens(tiny, T, first_id=10000 + T)
    out = torch.empty((T, WL.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, WL.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, WL.k), dtype=torch.float32, device="cuda")
    tiny.m.timing_enable(True)
    tiny.m.timing_reset()
    tiny.m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32)
    tiny.m.sync()
    kinds = tiny.m.timing()
    tiny.m.timing_enable(False)
    gemm = tiny.path == "tcgen05"
    assert kinds["gemm_gateup"][0] == (1 if gemm else 0)
    assert kinds["gemm_down"][0] == (1 if gemm else 0)
    assert kinds["expert_gateup"][0] == (0 if gemm else 1)
    ref = orc.moe_layer(tiny.layers[0], x)
    check_ids_weights(ids.cpu().numpy(), w.cpu().double().numpy(), ref["ids"], ref["w"])
    check_out(out32.cpu().double().numpy(), ref["out"])


def test_decode_batches_keep_gemv(tiny, torch):
    # T <= 8 never takes the GEMM
    T = 8
    x = draw_tokens(tiny, T, first_id=11000)
    out = torch.empty((T, WL.H), dtype=torch.int16, device="cuda")
    ids = torch.empty((T, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, WL.k), dtype=torch.float32, device="cuda")
    tiny.m.timing_enable(True)
    tiny.m.timing_reset()
    tiny.m.forward(to_dev_bf16(x), T, out, ids, w)
    tiny.m.sync()
    kinds = tiny.m.timing()
    tiny.m.timing_enable(False)
    assert kinds["gemm_gateup"][0] == 0 and kinds["expert_gateup"][0] == 1
