"""GPU parity of the stack workload: 8 Kimi-K3-shaped MoE layers resident in
HBM (~127 GB), each preceded by RMSNorm (eps 1e-6, unit gain) and followed by
a residual add, decoded at batch 1 and batch 4. Every token is drawn so that
its routing gap is >= 1e-3 at every layer (oracle logits).

Tolerances: ids bit-exact at every layer. Where both sides see the same
layer input — layer 0 of the stack, and every layer of the replay below,
which feeds the oracle the GPU's own layer inputs — the single-layer bars
hold: weights within 1e-5, layer output within relative L2 2e-3 and max-abs
1e-2 x RMS. The end-to-end output of L = 8 layers is the residual sum of the
layers' outputs, each allowed its own 2e-3 share, so it is held to L x the
single-layer bars (relative L2 1.6e-2, max-abs 8e-2 x RMS).

Through the whole stack the layer inputs themselves drift apart: the
residual stream is rounded to bf16 after every layer (|x| ~ 1e4, one bf16
ulp = 64), and where the GPU's fp32 sum and the oracle's double fall on
different sides of a rounding boundary (relative gap ~1e-6..1e-5 against an
ulp of 2^-8, i.e. ~0.1% of the elements) that element of the next
normalised input differs by one ulp (2^-8 relative). Each layer adds such
flips and propagates the earlier ones, so after several layers a logit can
move by ~1e-3, and the end-to-end weights of layers >= 1 are held to 1e-3.
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import (Setup, bits_to_f64, check_ids_weights, check_out,
                       draw_stack_token, to_dev_bf16)

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS[4]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def stack(torch):
    torch.cuda.empty_cache()
    s = Setup(WL, max_tokens=4)
    yield s
    s.close()
    torch.cuda.empty_cache()


def _forward(m, x, T, torch):
    out = torch.empty((T, WL.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, WL.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((WL.L, T, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((WL.L, T, WL.k), dtype=torch.float32, device="cuda")
    m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32)
    m.sync()
    return (out.cpu().numpy().view(np.uint16), out32.cpu().double().numpy(),
            ids.cpu().numpy(), w.cpu().double().numpy())


def test_rmsnorm_step(stack, torch):
    x = np.stack([synth.token(0, 4, 900 + t, WL.H) for t in range(3)])
    xn = torch.empty((3, WL.H), dtype=torch.int16, device="cuda")
    stack.m.step_rmsnorm(to_dev_bf16(x), 3, xn)
    torch.cuda.synchronize()
    got = xn.cpu().numpy().view(np.uint16)
    ref = orc.rmsnorm_bf16(x, WL.eps)
    diff = np.abs(bits_to_f64(got) - bits_to_f64(ref))
    ulp = np.abs(bits_to_f64(ref)) * 2.0 ** -7
    assert np.all(diff <= ulp + 1e-30)          # at most one bf16 ulp
    assert np.mean(got == ref) >= 0.999          # and almost always exact


@pytest.mark.parametrize("T", [1, 4])
def test_stack_decode(stack, torch, T):
    xs, refs = [], []
    for t in range(T):
        x, ref = draw_stack_token(stack, 1000 + 10 * T + t)
        xs.append(x)
        refs.append(ref)
    x = np.stack(xs)
    out, out32, ids, w = _forward(stack.m, x, T, torch)
    for t in range(T):
        for l in range(WL.L):
            check_ids_weights(ids[l, t:t + 1], w[l, t:t + 1], refs[t]["ids"][l],
                              refs[t]["w"][l], wtol=1e-5 if l == 0 else 1e-3)
    last = np.concatenate([r["last"] for r in refs])
    check_out(out32, last, rel_l2=WL.L * 2e-3, max_abs_rms=WL.L * 1e-2)
    # the bf16 output is the RNE rounding of the fp32 output
    rne = torch.from_numpy(out32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, rne)


def test_stack_matches_single_layer_composition(stack, torch):
    # layer l of the stack is exactly one MoE layer on bf16(rmsnorm(x)) with x
    # as the residual: check the first layer through the single-step calls
    x, ref = draw_stack_token(stack, 2000)
    xn = torch.empty((1, WL.H), dtype=torch.int16, device="cuda")
    stack.m.step_rmsnorm(to_dev_bf16(x[None, :]), 1, xn)
    torch.cuda.synchronize()
    xn_bits = xn.cpu().numpy().view(np.uint16)
    layer0 = orc.moe_layer(stack.layers[0], xn_bits, residual=x[None, :])
    assert sorted(layer0["ids"][0]) == sorted(ref["ids"][0, 0])


def test_stack_layers_on_gpu_inputs(stack, torch):
    """Replay the stack layer by layer on the GPU (same kernels, single-step
    calls) and compare every layer with the oracle on the GPU's own input."""
    x, _ = draw_stack_token(stack, 3000)
    H, k = WL.H, WL.k
    cur = x[None, :].copy()
    for l in range(WL.L):
        xn_d = torch.empty((1, H), dtype=torch.int16, device="cuda")
        stack.m.step_rmsnorm(to_dev_bf16(cur), 1, xn_d)
        logits = torch.empty((1, WL.E), dtype=torch.float32, device="cuda")
        stack.m.step_router(l, xn_d, 1, logits)
        ids = torch.empty((1, k), dtype=torch.int32, device="cuda")
        w = torch.empty((1, k), dtype=torch.float32, device="cuda")
        stack.m.step_topk(logits, 1, ids, w)
        hbuf = torch.empty((k, WL.I), dtype=torch.float32, device="cuda")
        stack.m.step_expert_gateup(l, xn_d, 1, ids, hbuf)
        y = torch.empty((1, H), dtype=torch.float32, device="cuda")
        stack.m.step_expert_down(l, hbuf, 1, ids, w, y)
        ysh = torch.empty((1, H), dtype=torch.float32, device="cuda")
        stack.m.step_shared(l, xn_d, 1, ysh)
        torch.cuda.synchronize()
        xn = xn_d.cpu().numpy().view(np.uint16)
        ref = orc.moe_layer(stack.layers[l], xn, residual=cur)
        check_ids_weights(ids.cpu().numpy(), w.cpu().double().numpy(), ref["ids"], ref["w"])
        yl = y.cpu().double().numpy() + ysh.cpu().double().numpy()
        check_out(yl, ref["routed"] + ref["shared"])
        # next layer input: the oracle's bf16 residual update of the GPU's sum
        nxt = bits_to_f64(cur) + yl
        cur = np.array([[orc.f64_to_bf16(v) for v in nxt[0]]], dtype=np.uint16)
