"""GPU parity at full Kimi-K3 layer size: hidden 7168, 896 MXFP4 experts
(17,547,264 B each, 15.7 GB resident), top-16, two bf16 shared experts.

Batch 1, batch 8 and batch 512 run on the same layer. The oracle computes
sampled tokens in full; routing (ids, weights) is checked for every token.
Tolerances as stated for the layer: ids bit-exact, weights 1e-5, output
relative L2 <= 2e-3 and max-abs <= 1e-2 x RMS. Steps: relative L2 <= 1e-5
(fp32 accumulation over <= 7168 exact-weight products).
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import (Setup, bits_to_f64, check_ids_weights, check_out,
                       draw_tokens, range_tokens, rel_l2, to_dev_bf16)

pytestmark = pytest.mark.gpu

WL1, WL2, WL3 = synth.WORKLOADS[1], synth.WORKLOADS[2], synth.WORKLOADS[3]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


# decode batches run the chain of kernels: router, then the routed and
# shared experts side by side in two phase kernels
@pytest.fixture(scope="module")
def k3(torch):
    s = Setup(WL1, max_tokens=512)
    yield s
    s.close()
    torch.cuda.empty_cache()


def _tokens(setup, wl, T, first_id=0):
    # tokens of workload wl's own stream on the shared K3 layer
    from moe_setup import gap_ok
    out = []
    for t in range(T):
        for r in range(synth.gen.REDRAWS_PER_TOKEN):
            x = synth.token(wl.seed, wl.cfg_id, first_id + t, wl.H, redraw=r)
            if gap_ok(orc.router_logits(setup.routers[0], x), wl.k):
                out.append(x)
                break
    return np.stack(out)


def _forward(m, x, T, torch, H=WL1.H, k=WL1.k):
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32)
    m.sync()
    return (out.cpu().numpy().view(np.uint16), out32.cpu().double().numpy(),
            ids.cpu().numpy(), w.cpu().double().numpy())


def test_span_size_and_layout_roundtrip(k3):
    assert k3.m.span_bytes == 17547264
    for e in (0, 1, 447, 895):
        back = np.empty(k3.m.span_bytes, dtype=np.uint8)
        k3.m.read_expert_span(0, e, back)
        assert np.array_equal(back, k3._span(0, e)), "expert %d" % e


def test_router_and_topk_steps(k3, torch):
    T = 8
    x = _tokens(k3, WL2, T, first_id=50)
    logits = torch.empty((T, WL1.E), dtype=torch.float32, device="cuda")
    k3.m.step_router(0, to_dev_bf16(x), T, logits)
    torch.cuda.synchronize()
    ref = orc.router_logits(k3.routers[0], x)
    assert np.max(np.abs(logits.cpu().double().numpy() - ref)) <= 1e-4
    ids = torch.empty((T, WL1.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, WL1.k), dtype=torch.float32, device="cuda")
    k3.m.step_topk(logits, T, ids, w)
    torch.cuda.synchronize()
    rid, rw = orc.topk_softmax(logits.cpu().double().numpy(), WL1.k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.max(np.abs(w.cpu().double().numpy() - rw)) <= 1e-6


def test_topk_step_ties(k3, torch):
    """Selection at full width (896 logits, top 16) with ties everywhere:
    equal logits go to the lower id, ids come out best first."""
    rng = np.random.default_rng(5)
    T = 9
    lg = rng.standard_normal((T, WL1.E)).astype(np.float32)
    lg[0, :] = 0.25                                   # all tied
    top = np.sort(lg[1])[::-1]
    lg[1, rng.permutation(WL1.E)[:40]] = top[15]      # 40 ties across the cut
    lg[2] = rng.integers(0, 5, WL1.E).astype(np.float32)  # five distinct values
    lg[3, WL1.E - 16:] = 9.0                          # the best are the last ids
    lg[4, :] = -np.inf
    lg[4, [895, 3, 500]] = [1.0, 1.0, 2.0]            # -inf fills the rest
    ids = torch.empty((T, WL1.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, WL1.k), dtype=torch.float32, device="cuda")
    k3.m.step_topk(torch.from_numpy(lg).cuda(), T, ids, w)
    torch.cuda.synchronize()
    rid, rw = orc.topk_softmax(lg.astype(np.float64), WL1.k)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.max(np.abs(w.cpu().double().numpy() - rw)) <= 1e-6


def test_expert_steps(k3, torch):
    T = 2
    x = _tokens(k3, WL2, T, first_id=60)
    rid, rw = orc.topk_softmax(orc.router_logits(k3.routers[0], x), WL1.k)
    hbuf = torch.empty((T * WL1.k, WL1.I), dtype=torch.float32, device="cuda")
    k3.m.step_expert_gateup(0, to_dev_bf16(x), T, torch.from_numpy(rid).cuda(), hbuf)
    torch.cuda.synchronize()
    got_h = hbuf.cpu().numpy()
    for (t, j) in [(0, 0), (0, 15), (1, 7)]:
        ref = orc.expert_gateup(k3._span(0, rid[t, j]), WL1.H, WL1.I, bits_to_f64(x[t]))
        assert rel_l2(got_h[t * WL1.k + j], ref) <= 1e-5
    # down step on the GPU's own h (as fp32) against the oracle on the same h
    y = torch.empty((T, WL1.H), dtype=torch.float32, device="cuda")
    w32 = rw.astype(np.float32)
    k3.m.step_expert_down(0, hbuf, T, torch.from_numpy(rid).cuda(),
                          torch.from_numpy(w32).cuda(), y)
    torch.cuda.synchronize()
    t = 1
    ref = sum(np.float64(w32[t, j]) * orc.expert_down(k3._span(0, rid[t, j]), WL1.H, WL1.I,
                                                      got_h[t * WL1.k + j].astype(np.float64))
              for j in range(WL1.k))
    assert rel_l2(y.cpu().double().numpy()[t], ref) <= 1e-5


def test_shared_step(k3, torch):
    x = _tokens(k3, WL2, 1, first_id=70)
    y = torch.empty((1, WL1.H), dtype=torch.float32, device="cuda")
    k3.m.step_shared(0, to_dev_bf16(x), 1, y)
    torch.cuda.synchronize()
    ref = sum(orc.shared_ffn(*s, bits_to_f64(x[0])) for s in k3.shared[0])
    # the shared part is ~1e-5 of the routed part in the full layer, so it
    # gets its own check here
    assert rel_l2(y.cpu().double().numpy()[0], ref) <= 1e-5


def test_decode_batch1(k3, torch):
    x = _tokens(k3, WL1, 3)
    for t in range(3):
        out, out32, ids, w = _forward(k3.m, x[t:t + 1], 1, torch)
        ref = orc.moe_layer(k3.layers[0], x[t:t + 1])
        check_ids_weights(ids, w, ref["ids"], ref["w"])
        check_out(out32, ref["out"])


def test_decode_batch8(k3, torch):
    x = _tokens(k3, WL2, 8)
    out, out32, ids, w = _forward(k3.m, x, 8, torch)
    ref = orc.moe_layer(k3.layers[0], x)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


def test_prefill_batch512(k3, torch):
    T = 512
    x = _tokens(k3, WL3, T)
    out, out32, ids, w = _forward(k3.m, x, T, torch)
    rid, rw = orc.topk_softmax(orc.router_logits(k3.routers[0], x), WL1.k)
    check_ids_weights(ids, w, rid, rw)          # every token's routing
    # full outputs on every eighth token and the last one (65 of 512)
    sample = list(range(0, T, 8)) + [T - 1]
    ref = orc.moe_layer(k3.layers[0], x[sample])
    check_out(out32[sample], ref["out"])
    # and every token's output is finite with the bf16 output its rounding
    assert np.all(np.isfinite(out32))
    rne = torch.from_numpy(out32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, rne)


@pytest.mark.parametrize("T", [1, 8, 16])
def test_input_range(k3, torch, T):
    """Hidden states at the edges of the range: a token scaled by 2^20, one
    by 2^-60, one with a 2^20 chunk and a 2^-40 chunk. T = 1 runs each on
    its own (the decode chain), T = 8 and T = 16 mix them with N(0,1)
    tokens (decode batch and the tcgen05 batch path)."""
    xs = range_tokens(k3, first_id=60000)
    if T > 1:
        xs = np.concatenate([xs, _tokens(k3, WL2, T - 3, first_id=60100)])
    batches = [xs[i:i + 1] for i in range(3)] if T == 1 else [xs]
    for x in batches:
        n = x.shape[0]
        out, out32, ids, w = _forward(k3.m, x, n, torch)
        assert np.all(np.isfinite(out32))
        ref = orc.moe_layer(k3.layers[0], x)
        check_ids_weights(ids, w, ref["ids"], ref["w"])
        check_out(out32, ref["out"])


def test_ragged_batch(k3, torch):
    T = 5
    x = _tokens(k3, WL2, T, first_id=500)
    out, out32, ids, w = _forward(k3.m, x, T, torch)
    ref = orc.moe_layer(k3.layers[0], x)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


def _bf16_rne(v):
    """float64 array -> bf16 bits, round to nearest even through fp32."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_verify_pass_t2(k3, torch):
    """A two-position verify call (n-gram speculation checks a drafted token
    in the same pass as the current one [Deltafin README, "N-gram
    speculation"]). The drafted position's hidden state is correlated with
    the first (0.8 x1 + 0.6 z), so the two top-16 sets overlap and the
    shared experts are read once for both positions."""
    from moe_setup import gap_ok
    x1 = _tokens(k3, WL1, 1, first_id=900)[0]
    for r in range(synth.gen.REDRAWS_PER_TOKEN):
        z = synth.token(WL1.seed, WL1.cfg_id, 901, WL1.H, redraw=r)
        x2 = _bf16_rne(0.8 * bits_to_f64(x1) + 0.6 * bits_to_f64(z))
        if gap_ok(orc.router_logits(k3.routers[0], x2[None]), WL1.k):
            break
    x = np.stack([x1, x2])
    out, out32, ids, w = _forward(k3.m, x, 2, torch)
    ref = orc.moe_layer(k3.layers[0], x)
    shared = len(set(ref["ids"][0]) & set(ref["ids"][1]))
    assert shared >= 2, "the drafted position shares %d experts" % shared
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


def test_graph_replay_matches_eager(k3, torch):
    """df_moe_graph_*: a forward pass captured once and replayed on new
    contents of its input buffer gives, bit for bit, the eager call's
    results (the same kernels), and the oracle's routing."""
    import mxfp4_routed_expert_top_gb300 as dfm
    x = _tokens(k3, WL1, 3, first_id=1300)
    x_buf = torch.empty((1, WL1.H), dtype=torch.int16, device="cuda")
    out = torch.empty((1, WL1.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((1, WL1.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((1, WL1.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, WL1.k), dtype=torch.float32, device="cuda")
    g = k3.m.graph(x_buf, 1, out, ids, w, out_f32=out32)
    try:
        assert g.launch_count() >= 3
        for t in range(3):
            x_buf.copy_(to_dev_bf16(x[t:t + 1]))
            g.launch()
            torch.cuda.synchronize()
            got = (out.cpu().numpy().copy(), out32.cpu().numpy().copy(), ids.cpu().numpy().copy(),
                   w.cpu().numpy().copy())
            e_out, e_out32, e_ids, e_w = _forward(k3.m, x[t:t + 1], 1, torch)
            assert np.array_equal(got[0].view(np.uint16), e_out)
            assert np.array_equal(got[1], e_out32.astype(np.float32))
            assert np.array_equal(got[2], e_ids)
            assert np.array_equal(got[3], e_w.astype(np.float32))
            rid, rw = orc.topk_softmax(orc.router_logits(k3.routers[0], x[t:t + 1]), WL1.k)
            check_ids_weights(got[2], got[3].astype(np.float64), rid, rw)
    finally:
        g.close()


def test_stream_read_probe(torch):
    """df_moe_stream_read reads every 16-byte word exactly once: the XOR of
    its per-thread words is the XOR of the buffer's words."""
    import mxfp4_routed_expert_top_gb300 as dfm
    n = (64 << 20) + 48  # not a multiple of the grid's stride
    buf = torch.zeros(n // 4, dtype=torch.int32, device="cuda")
    buf[12345] = 0x1234567
    buf[n // 4 - 1] = 0x70000001
    sink = torch.empty(8 * torch.cuda.get_device_properties(0).multi_processor_count * 256,
                       dtype=torch.int32, device="cuda")
    dfm.stream_read(buf, n, sink)
    torch.cuda.synchronize()
    # the probe writes 4 * SMs * 256 words; the rest of sink is never read
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    folded = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32)[:4 * nsm * 256])
    assert folded == (0x1234567 ^ 0x70000001)
    with pytest.raises(dfm.DfMoeError):
        dfm.stream_read(buf, n - 4, sink)
