"""GPU parity on the tiny workload (H=256, I=64, 8 experts, top-2, one shared
expert): every step of the hot path through the C ABI against the oracle,
the whole layer, edge and degenerate cases, errors and determinism.

Step tolerances: the kernels accumulate in fp32 over at most a few thousand
products of exactly-representable weights, so a relative L2 error of 1e-5
leaves a wide margin over fp32 rounding (~sqrt(K) * 2^-24 ~ 1e-6). The
layer-output bar is the stated one: relative L2 <= 2e-3 and max-abs error
<= 1e-2 x output RMS; ids bit-exact as sets, weights within 1e-5.
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import (Setup, bits_to_f64, check_ids_weights, check_out,
                       draw_tokens, range_tokens, rel_l2, to_dev_bf16)

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS[0]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def tiny(torch):
    s = Setup(WL, max_tokens=16)
    yield s
    s.close()


def test_device_generator_matches_host(torch):
    n, H, I = 3, WL.H, WL.I
    span = synth.span_bytes(H, I)
    buf = torch.empty(n * span, dtype=torch.uint8, device="cuda")
    synth.dev_expert_spans(WL.seed, WL.wcfg, 0, 2, n, H, I, buf.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    host = synth.expert_spans(WL.seed, WL.wcfg, 0, 2, n, H, I)
    assert np.array_equal(buf.cpu().numpy().reshape(n, span), host)


def test_layout_roundtrip(tiny):
    span = tiny.m.span_bytes
    assert span == synth.span_bytes(WL.H, WL.I)
    for e in range(WL.E):
        back = np.empty(span, dtype=np.uint8)
        tiny.m.read_expert_span(0, e, back)
        assert np.array_equal(back, tiny._span(0, e)), "expert %d" % e


def test_router_step(tiny, torch):
    x = draw_tokens(tiny, 5)
    logits = torch.empty((5, WL.E), dtype=torch.float32, device="cuda")
    tiny.m.step_router(0, to_dev_bf16(x), 5, logits)
    torch.cuda.synchronize()
    ref = orc.router_logits(tiny.routers[0], x)
    assert np.max(np.abs(logits.cpu().double().numpy() - ref)) <= 1e-5


def test_topk_step(tiny, torch):
    rng = np.random.default_rng(11)
    T = 9
    lg = rng.standard_normal((T, WL.E)).astype(np.float32)
    lg[0, :] = 0.5  # all tied: the lowest ids win, in order
    ids = torch.empty((T, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, WL.k), dtype=torch.float32, device="cuda")
    tiny.m.step_topk(torch.from_numpy(lg).cuda(), T, ids, w)
    torch.cuda.synchronize()
    rid, rw = orc.topk_softmax(lg.astype(np.float64), WL.k)
    assert np.array_equal(ids.cpu().numpy(), rid)  # order too: same fp32 inputs
    assert np.max(np.abs(w.cpu().double().numpy() - rw)) <= 1e-6


@pytest.mark.parametrize("T", [1, 2, 9, 16])
def test_group_step(tiny, torch, T):
    rng = np.random.default_rng(T)
    ids = np.stack([rng.permutation(WL.E)[:WL.k] for _ in range(T)]).astype(np.int32)
    offs = torch.empty(WL.E + 1, dtype=torch.int32, device="cuda")
    tok = torch.empty(T * WL.k, dtype=torch.int32, device="cuda")
    slot = torch.empty(T * WL.k, dtype=torch.int32, device="cuda")
    nu = torch.empty(1, dtype=torch.int32, device="cuda")
    tiny.m.step_group(torch.from_numpy(ids).cuda(), T, offs, tok, slot, nu)
    torch.cuda.synchronize()
    roffs, rtok, rslot, rn = orc.group(ids, WL.E)
    assert np.array_equal(offs.cpu().numpy(), roffs)
    assert np.array_equal(tok.cpu().numpy(), rtok)
    assert np.array_equal(slot.cpu().numpy(), rslot)
    assert nu.item() == rn


@pytest.mark.parametrize("T, hot", [(512, False), (600, False), (600, True)])
def test_group_step_large(torch, T, hot):
    """Grouping of many assignments (64 experts, top-16): up to 8192 sort in
    shared memory, more in place in global memory (600 x 16 = 9600); a hot
    expert in every token's first slot gives the longest segment."""
    import mxfp4_routed_expert_top_gb300 as dfm
    E, k = 64, 16
    rng = np.random.default_rng(T + hot)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    if hot:
        for t in range(T):
            row = [3] + [e for e in ids[t] if e != 3][:k - 1]
            ids[t] = row
    with dfm.MoE(WL.H, E, k, WL.I, WL.n_shared, WL.Is, max_tokens=T) as m:
        offs = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        tok = torch.empty(T * k, dtype=torch.int32, device="cuda")
        slot = torch.empty(T * k, dtype=torch.int32, device="cuda")
        nu = torch.empty(1, dtype=torch.int32, device="cuda")
        m.step_group(torch.from_numpy(ids).cuda(), T, offs, tok, slot, nu)
        torch.cuda.synchronize()
        roffs, rtok, rslot, rn = orc.group(ids, E)
        assert np.array_equal(offs.cpu().numpy(), roffs)
        assert np.array_equal(tok.cpu().numpy(), rtok)
        assert np.array_equal(slot.cpu().numpy(), rslot)
        assert nu.item() == rn


def _oracle_route(tiny, x):
    return orc.topk_softmax(orc.router_logits(tiny.routers[0], x), WL.k)


@pytest.mark.parametrize("T", [1, 3])
def test_gateup_step(tiny, torch, T):
    x = draw_tokens(tiny, T, first_id=100)
    rid, _ = _oracle_route(tiny, x)
    hbuf = torch.empty((T * WL.k, WL.I), dtype=torch.float32, device="cuda")
    tiny.m.step_expert_gateup(0, to_dev_bf16(x), T, torch.from_numpy(rid).cuda(), hbuf)
    torch.cuda.synchronize()
    got = hbuf.cpu().double().numpy()
    for t in range(T):
        for j in range(WL.k):
            ref = orc.expert_gateup(tiny._span(0, rid[t, j]), WL.H, WL.I, bits_to_f64(x[t]))
            assert rel_l2(got[t * WL.k + j], ref) <= 1e-5


@pytest.mark.parametrize("T", [1, 3])
def test_down_step(tiny, torch, T):
    x = draw_tokens(tiny, T, first_id=200)
    rid, rw = _oracle_route(tiny, x)
    h = np.stack([orc.expert_gateup(tiny._span(0, rid[t, j]), WL.H, WL.I, bits_to_f64(x[t]))
                  for t in range(T) for j in range(WL.k)]).astype(np.float32)
    y = torch.empty((T, WL.H), dtype=torch.float32, device="cuda")
    tiny.m.step_expert_down(0, torch.from_numpy(h).cuda(), T, torch.from_numpy(rid).cuda(),
                            torch.from_numpy(rw.astype(np.float32)).cuda(), y)
    torch.cuda.synchronize()
    got = y.cpu().double().numpy()
    for t in range(T):
        ref = sum(np.float64(np.float32(rw[t, j])) *
                  orc.expert_down(tiny._span(0, rid[t, j]), WL.H, WL.I,
                                  h[t * WL.k + j].astype(np.float64))
                  for j in range(WL.k))
        assert rel_l2(got[t], ref) <= 1e-5


def test_shared_step(tiny, torch):
    x = draw_tokens(tiny, 2, first_id=300)
    y = torch.empty((2, WL.H), dtype=torch.float32, device="cuda")
    tiny.m.step_shared(0, to_dev_bf16(x), 2, y)
    torch.cuda.synchronize()
    for t in range(2):
        ref = sum(orc.shared_ffn(*s, bits_to_f64(x[t])) for s in tiny.shared[0])
        assert rel_l2(y.cpu().double().numpy()[t], ref) <= 1e-5


def _forward(m, x, T, torch, residual=None, L=1, k=WL.k, H=WL.H):
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((L, T, k), dtype=torch.float32, device="cuda")
    m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32,
              residual=None if residual is None else to_dev_bf16(residual))
    m.sync()
    return (out.cpu().numpy().view(np.uint16), out32.cpu().double().numpy(),
            ids.cpu().numpy(), w.cpu().double().numpy())


@pytest.mark.parametrize("T", [1, 2, 7, 16])
def test_forward_matches_oracle(tiny, torch, T):
    x = draw_tokens(tiny, T, first_id=1000 + 20 * T)
    res = np.stack([synth.token(WL.seed, WL.cfg_id, 5000 + t, WL.H,
                                kind=synth.gen.KIND_RESIDUAL) for t in range(T)])
    out, out32, ids, w = _forward(tiny.m, x, T, torch, residual=res)
    ref = orc.moe_layer(tiny.layers[0], x, residual=res)
    check_ids_weights(ids[0], w[0], ref["ids"], ref["w"])
    check_out(out32, ref["out"])
    # the bf16 output is the RNE rounding of the fp32 output
    rne = torch.from_numpy(out32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, rne)


def test_forward_host_buffers(tiny, torch):
    T = 3
    x = draw_tokens(tiny, T, first_id=7000)
    out = np.empty((T, WL.H), dtype=np.uint16)
    out32 = np.empty((T, WL.H), dtype=np.float32)
    ids = np.empty((T, WL.k), dtype=np.int32)
    w = np.empty((T, WL.k), dtype=np.float32)
    tiny.m.forward_host(x, T, out, ids=ids, weights=w, out_f32=out32)
    ref = orc.moe_layer(tiny.layers[0], x)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


@pytest.mark.parametrize("kind", ["numpy", "pinned", "device", "mixed"])
@pytest.mark.parametrize("T", [3, 12])
def test_forward_host_buffer_kinds(tiny, torch, kind, T):
    """The host-buffer forward moves data on the device where it can (pinned
    host memory: a copy kernel in, the last kernel writes out), through a
    staging copy for ordinary host memory, by cudaMemcpyAsync for device
    memory; every way gives the device forward's bits."""
    x = draw_tokens(tiny, T, first_id=7300 + T)
    d = [torch.empty((T, WL.H), dtype=torch.int16, device="cuda"),
         torch.empty((T, WL.H), dtype=torch.float32, device="cuda"),
         torch.empty((T, WL.k), dtype=torch.int32, device="cuda"),
         torch.empty((T, WL.k), dtype=torch.float32, device="cuda")]
    tiny.m.forward(to_dev_bf16(x), T, d[0], d[2], d[3], out_f32=d[1])
    tiny.m.sync()
    want = [t.cpu().numpy() for t in d]   # the device forward's out, out32, ids, w

    def buf(shape, dtype, k):
        a = np.zeros(shape, dtype=dtype)
        if k == "numpy":
            return a, lambda b: b
        t = torch.from_numpy(a)
        t = t.pin_memory() if k == "pinned" else t.cuda()
        return t, lambda b: b.cpu().numpy()
    kinds = {"mixed": ["pinned", "numpy", "device", "pinned", "numpy"]}.get(kind, [kind] * 5)
    xb, _ = buf((T, WL.H), np.int16, kinds[0])
    if kind == "numpy" or kinds[0] == "numpy":
        xb[...] = x.view(np.int16)
    else:
        xb.copy_(torch.from_numpy(x.view(np.int16)))
    out, g0 = buf((T, WL.H), np.int16, kinds[1])
    out32, g1 = buf((T, WL.H), np.float32, kinds[2])
    ids, g2 = buf((T, WL.k), np.int32, kinds[3])
    w, g3 = buf((T, WL.k), np.float32, kinds[4])
    tiny.m.forward_host(xb, T, out, ids=ids, weights=w, out_f32=out32)
    got = (g0(out), g1(out32), g2(ids), g3(w))
    for a, b in zip(got, want):
        assert a.shape == b.shape and a.dtype == b.dtype
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_forward_is_deterministic(tiny, torch):
    x = draw_tokens(tiny, 16, first_id=8000)
    a = _forward(tiny.m, x, 16, torch)
    b = _forward(tiny.m, x, 16, torch)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_errors(tiny, torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    x = to_dev_bf16(draw_tokens(tiny, 1, first_id=9000))
    out = torch.empty((1, WL.H), dtype=torch.int16, device="cuda")
    ids = torch.empty((1, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, WL.k), dtype=torch.float32, device="cuda")
    for T in (0, 17, -1):
        with pytest.raises(dfm.DfMoeError) as ei:
            tiny.m.forward(x, T, out, ids, w)
        assert ei.value.code == -5
    with pytest.raises(dfm.DfMoeError) as ei:
        tiny.m.forward(x, 1, None, ids, w)
    assert ei.value.code == -1
    # device arrays of the steps off a 16-byte boundary: refused before any
    # launch (the kernels read them with vector accesses)
    flat = torch.zeros(2 * WL.H + 8, dtype=torch.int16, device="cuda")
    xm = flat[1:1 + WL.H]
    lg = torch.empty((1, WL.E), dtype=torch.float32, device="cuda")
    hb = torch.empty((WL.k, WL.I), dtype=torch.float32, device="cuda")
    ysh = torch.empty((1, WL.H), dtype=torch.float32, device="cuda")
    for call in (lambda: tiny.m.step_router(0, xm, 1, lg),
                 lambda: tiny.m.step_expert_gateup(0, xm, 1, ids, hb),
                 lambda: tiny.m.step_shared(0, xm, 1, ysh),
                 lambda: tiny.m.step_rmsnorm(xm, 1, flat[8:8 + WL.H])):
        with pytest.raises(dfm.DfMoeError) as ei:
            call()
        assert ei.value.code == -1
    with dfm.MoE(WL.H, WL.E, WL.k, WL.I, WL.n_shared, WL.Is) as fresh:
        with pytest.raises(dfm.DfMoeError) as ei:
            fresh.forward(x, 1, out, ids, w)
        assert ei.value.code == -4  # nothing loaded yet
        with pytest.raises(dfm.DfMoeError) as ei:
            fresh.load_experts(1, router=tiny.routers[0])
        assert ei.value.code == -5  # no layer 1
    with pytest.raises(dfm.DfMoeError) as ei:
        dfm.MoE(WL.H + 1, WL.E, WL.k, WL.I, WL.n_shared, WL.Is)
    assert ei.value.code == -1


def _host_handle(torch, spans, router, shared, k=WL.k, n_shared=WL.n_shared, T=4):
    import mxfp4_routed_expert_top_gb300 as dfm
    m = dfm.MoE(WL.H, WL.E, k, WL.I, n_shared, WL.Is, max_tokens=T)
    m.load_experts(0, router=router, experts=spans, expert_begin=0, expert_count=WL.E,
                   shared=shared if n_shared else None)
    return m


def test_all_zero_codes_leave_shared_only(tiny, torch):
    spans = synth.expert_spans(WL.seed, WL.wcfg, 0, 0, WL.E, WL.H, WL.I)
    q = WL.H * WL.I // 2
    s = WL.H * WL.I // 32
    for e in range(WL.E):
        spans[e, 0:q] = 0
        spans[e, q + s:2 * q + s] = 0
        spans[e, 2 * q + 2 * s:3 * q + 2 * s] = 0
    x = draw_tokens(tiny, 2, first_id=9100)
    with _host_handle(torch, spans, tiny.routers[0], tiny.shared[0]) as m:
        out, out32, ids, w = _forward(m, x, 2, torch)
    for t in range(2):
        ref = orc.shared_ffn(*tiny.shared[0][0], bits_to_f64(x[t]))
        assert rel_l2(out32[t], ref) <= 1e-5


def test_single_nonzero_code_pins_nibble_order(tiny, torch):
    # one gate weight and one up weight non-zero: g and u each pick one x
    spans = np.zeros((WL.E, synth.span_bytes(WL.H, WL.I)), dtype=np.uint8)
    q, s = WL.H * WL.I // 2, WL.H * WL.I // 32
    spans[:, q:q + s] = 127
    spans[:, 2 * q + s:2 * q + 2 * s] = 127
    spans[:, 3 * q + 2 * s:] = 127
    row, col = 5, 33  # odd column -> high nibble
    for e in range(WL.E):
        spans[e, row * (WL.H // 2) + col // 2] = 0x20          # gate[5][33] = 1.0
        spans[e, q + s + row * (WL.H // 2) + col // 2] = 0x20  # up[5][33] = 1.0
        # down[9][5] = 1.0 (even column -> low nibble)
        spans[e, 2 * q + 2 * s + 9 * (WL.I // 2) + 5 // 2] = 0x20 if 5 % 2 else 0x02
    x = draw_tokens(tiny, 1, first_id=9200)
    with _host_handle(torch, spans, tiny.routers[0], None, n_shared=0) as m:
        out, out32, ids, w = _forward(m, x, 1, torch)
    xv = bits_to_f64(x[0])[col]
    h = xv / (1 + np.exp(-xv)) * xv
    expect = np.zeros(WL.H)
    expect[9] = h  # every expert gives the same y; weights sum to 1
    assert np.allclose(out32[0], expect, rtol=1e-5, atol=1e-6 * abs(h) + 1e-30)


def test_k_equals_e_and_no_shared(tiny, torch):
    spans = synth.expert_spans(WL.seed, WL.wcfg, 0, 0, WL.E, WL.H, WL.I)
    x = draw_tokens(tiny, 2, first_id=9300)
    with _host_handle(torch, spans, tiny.routers[0], None, k=WL.E, n_shared=0) as m:
        out, out32, ids, w = _forward(m, x, 2, torch, k=WL.E)
    L = orc.Layer(WL.H, WL.E, WL.E, WL.I, WL.Is, tiny.routers[0], [],
                  lambda l, e: spans[e])
    ref = orc.moe_layer(L, x)
    check_ids_weights(ids[0], w[0], ref["ids"], ref["w"])
    check_out(out32, ref["out"])


@pytest.mark.parametrize("T", [1, 2])
def test_one_token_selects_in_the_gateup_phase(tiny, torch, T):
    """One token: the gate/up phase kernel selects the experts itself (no
    top-k or grouping launch); two and more take the top-k and grouping
    kernels. Both against the oracle, with the ids and weights the
    selection publishes."""
    x = draw_tokens(tiny, T, first_id=12000 + 10 * T)
    out32 = torch.empty((T, WL.H), dtype=torch.float32, device="cuda")
    out = torch.empty((T, WL.H), dtype=torch.int16, device="cuda")
    ids = torch.empty((T, WL.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, WL.k), dtype=torch.float32, device="cuda")
    tiny.m.timing_enable(True)
    tiny.m.timing_reset()
    tiny.m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32)
    tiny.m.sync()
    kinds = tiny.m.timing()
    tiny.m.timing_enable(False)
    separate = 0 if T == 1 else 1
    assert kinds["topk"][0] == separate and kinds["group"][0] == separate
    assert kinds["expert_gateup"][0] == 1
    ref = orc.moe_layer(tiny.layers[0], x)
    check_ids_weights(ids.cpu().numpy(), w.cpu().double().numpy(), ref["ids"], ref["w"])
    check_out(out32.cpu().double().numpy(), ref["out"])


# ---- the input range of the decode paths ----------------------------------
# A hidden state may hold any bf16 value. The decode GEMVs multiply x as f16
# after scaling each (token, 512-column chunk) by a power of two, so large
# (2^20 ~ 1e6) and small (2^-60 ~ 1e-18) tokens are exact as well. Scaling a
# token by a power of two scales its logits exactly, so tokens that pass the
# gap rule still do; the mixed token is checked on its own.

@pytest.mark.parametrize("T", [1, 3, 9])
def test_forward_input_range(tiny, torch, T):
    """Decode batches (T = 1 for each token, T = 3 for all three) and the
    batch path (T = 9: the three tokens and six N(0,1) ones)."""
    xs = range_tokens(tiny, first_id=30000)
    if T == 9:
        xs = np.concatenate([xs, draw_tokens(tiny, 6, first_id=30100)])
    batches = [xs[i:i + 1] for i in range(3)] if T == 1 else [xs]
    for x in batches:
        n = x.shape[0]
        out, out32, ids, w = _forward(tiny.m, x, n, torch)
        assert np.all(np.isfinite(out32))
        ref = orc.moe_layer(tiny.layers[0], x)
        check_ids_weights(ids[0], w[0], ref["ids"], ref["w"])
        check_out(out32, ref["out"])


def test_gateup_step_input_range(tiny, torch):
    """The gate/up step on its own at the single-step bar (1e-5)."""
    x = range_tokens(tiny, first_id=30200)
    rid, _ = _oracle_route(tiny, x)
    hbuf = torch.empty((3 * WL.k, WL.I), dtype=torch.float32, device="cuda")
    tiny.m.step_expert_gateup(0, to_dev_bf16(x), 3, torch.from_numpy(rid).cuda(), hbuf)
    torch.cuda.synchronize()
    got = hbuf.cpu().double().numpy()
    for t in range(3):
        for j in range(WL.k):
            ref = orc.expert_gateup(tiny._span(0, rid[t, j]), WL.H, WL.I, bits_to_f64(x[t]))
            assert rel_l2(got[t * WL.k + j], ref) <= 1e-5


# ---- E8M0 codes 0 and 255 -------------------------------------------------
# The generator never draws them (scales are 2^-8 .. 2^0). The oracle decodes
# them as the format defines them, 2^-127 and NaN. The decode GEMVs read code
# 0 as 0 (a block of 2^-127 weights adds below 1e-37 here, invisible at the
# stated bars) and code 255 as +inf: every output that the oracle makes NaN
# comes out non-finite.

def _gate_scale_offset(row, block):
    q = WL.H * WL.I // 2
    return q + row * (WL.H // 32) + block


def test_e8m0_code_zero(tiny, torch):
    spans = synth.expert_spans(WL.seed, WL.wcfg, 0, 0, WL.E, WL.H, WL.I)
    for e in range(WL.E):
        for row in (0, 7, 33):
            spans[e, _gate_scale_offset(row, 2)] = 0
    x = draw_tokens(tiny, 2, first_id=30300)
    with _host_handle(torch, spans, tiny.routers[0], tiny.shared[0]) as m:
        out, out32, ids, w = _forward(m, x, 2, torch)
    L = orc.Layer(WL.H, WL.E, WL.k, WL.I, WL.Is, tiny.routers[0], tiny.shared[0],
                  lambda l, e: spans[e])
    ref = orc.moe_layer(L, x)
    check_ids_weights(ids[0], w[0], ref["ids"], ref["w"])
    check_out(out32, ref["out"])


def test_e8m0_code_255(tiny, torch):
    spans = synth.expert_spans(WL.seed, WL.wcfg, 0, 0, WL.E, WL.H, WL.I)
    for e in range(WL.E):
        spans[e, _gate_scale_offset(3, 1)] = 255
    x = draw_tokens(tiny, 1, first_id=30400)
    with _host_handle(torch, spans, tiny.routers[0], tiny.shared[0]) as m:
        out, out32, ids, w = _forward(m, x, 1, torch)
    L = orc.Layer(WL.H, WL.E, WL.k, WL.I, WL.Is, tiny.routers[0], tiny.shared[0],
                  lambda l, e: spans[e])
    ref = orc.moe_layer(L, x)
    nan = np.isnan(ref["out"])
    assert nan.any()
    assert not np.any(np.isfinite(out32[nan]))
    assert np.array_equal(np.isfinite(out32), ~nan)
