"""The MXFP8-activation variant (DF_MOE_MXFP8_ACT) against the oracle.

Kimi K3 is trained with MXFP8 activations (Deltafin analysis, section 2.1);
the variant rounds the routed experts' inputs to that format and runs the
block-scaled MXFP4 x MXFP8 MMA of the 5th-generation tensor cores. The
rounding is a decision (a quantised code), so the checks take it on the same
values on both sides:
  * the library's rounding routine is bit-exact with the oracle's on fp32
    rows, edge cases included;
  * gate/up: h before its rounding matches the oracle's gate/up on the
    oracle's MXFP8 rounding of x (the same codes: x is exact in fp32), at the
    GEMM tolerance 1e-5 (relative L2 per assignment: products are exact, the
    sums fp32);
  * down: the library rounds the given h and matches the oracle's down on the
    oracle's rounding of the same h, 1e-5;
  * the layer: forward matches the oracle's MXFP8 layer fed with the h of the
    library's own gate/up GEMM (the same kernel on the same inputs), at the
    layer bars; ids and routing weights are the exact path's. The error
    against the exact layer is reported separately and bounded loosely (the
    format keeps 4 significant bits: a few per cent).
Shapes: a small layer (H = 256, I = 128, 8 experts, top-2) with a hot expert
that needs two token passes, and the K3 layer at batch 1 and 512.
"""
import numpy as np
import pytest

import oracle as orc
import synth
from synth.workloads import Workload
from moe_setup import Setup, check_ids_weights, check_out, draw_tokens, rel_l2, to_dev_bf16

pytestmark = pytest.mark.gpu

SMALL = Workload("small-h256-i128-e8-top2", 5, H=256, I=128, E=8, k=2, n_shared=1, Is=64, T=1)
K3 = synth.WORKLOADS[3]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


@pytest.fixture(scope="module")
def small(torch):
    s = Setup(SMALL, max_tokens=160, mxfp8=True)
    yield s
    s.close()


def x_f64(x):
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def test_rounding_matches_oracle(small, torch):
    rng = np.random.default_rng(3)
    rows, n = 40, 256
    v = (rng.standard_normal((rows, n)) *
         np.ldexp(1.0, rng.integers(-40, 40, (rows, 1)))).astype(np.float32)
    v[0, :32] = 0.0                                   # an all-zero block
    v[1, :32] = 448.0 * 2.0 ** -3                     # a constant block
    v[2, 5] = 3e38                                    # near the float maximum
    v[3, :32] = np.float32(1e-41)                     # subnormal floats
    v[4, :32] = rng.standard_normal(32) * 1e-39       # mixed subnormal block
    # every E4M3 midpoint at unit scale (ties to even), both signs
    mids = np.array([(orc.e4m3_value(c) + orc.e4m3_value(c + 1)) / 2 for c in range(0x7E)])
    blk = np.concatenate([mids, -mids, [448.0, 460.0, 464.0, 500.0]])
    for i in range(0, len(blk) - 31, 31):
        r = 5 + i // 31
        v[r, :31] = blk[i:i + 31]
        v[r, 31] = 256.0                              # keeps the block exponent at 0
    vd = torch.from_numpy(v).cuda()
    codes = torch.empty((rows, n), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, n // 32), dtype=torch.uint8, device="cuda")
    small.m.step_mxfp8(vd, rows, n, codes, scales)
    torch.cuda.synchronize()
    rc, rs = orc.mxfp8_quantize(v.astype(np.float64))
    assert np.array_equal(scales.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_span_round_trip(small, torch):
    for e in (0, 3, 7):
        got = np.empty(small.m.span_bytes, dtype=np.uint8)
        small.m.read_expert_span(0, e, got)
        assert np.array_equal(got, small._span(0, e))


def _ids_hot(T, k, E, hot, seed):
    """Assignments with expert `hot` in every token's first slot (a hot
    expert with T tokens), the rest drawn without repeats."""
    rng = np.random.default_rng(seed)
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        others = [e for e in rng.permutation(E) if e != hot][:k - 1]
        ids[t] = [hot] + others
    return ids


@pytest.mark.parametrize("T", [1, 7, 100])
def test_gateup_step(small, torch, T):
    wl = SMALL
    x = np.stack([synth.token(wl.seed, wl.cfg_id, 300 + t, wl.H) for t in range(T)])
    ids = _ids_hot(T, wl.k, wl.E, hot=3, seed=T)   # expert 3: T tokens (two passes at 100)
    hbuf = torch.zeros((T * wl.k, wl.I), dtype=torch.float32, device="cuda")
    small.m.step_expert_gateup(0, to_dev_bf16(x), T, torch.from_numpy(ids).cuda(), hbuf)
    torch.cuda.synchronize()
    got = hbuf.cpu().numpy().astype(np.float64)
    xq = orc.mxfp8_round(x_f64(x))
    for t in range(T):
        for j in range(wl.k):
            ref = orc.expert_gateup(small._span(0, int(ids[t, j])), wl.H, wl.I, xq[t])
            assert rel_l2(got[t * wl.k + j], ref) <= 1e-5, (t, j)


@pytest.mark.parametrize("T", [1, 9, 100])
def test_down_step(small, torch, T):
    wl = SMALL
    rng = np.random.default_rng(40 + T)
    h = (rng.standard_normal((T * wl.k, wl.I)) *
         np.ldexp(1.0, rng.integers(-6, 6, (T * wl.k, 1)))).astype(np.float32)
    ids = _ids_hot(T, wl.k, wl.E, hot=6, seed=100 + T)
    w = rng.uniform(0.1, 1.0, (T, wl.k)).astype(np.float32)
    y = torch.zeros((T, wl.H), dtype=torch.float32, device="cuda")
    small.m.step_expert_down(0, torch.from_numpy(h).cuda(), T, torch.from_numpy(ids).cuda(),
                             torch.from_numpy(w).cuda(), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    hq = orc.mxfp8_round(h.astype(np.float64))
    for t in range(T):
        ref = sum(float(w[t, j]) * orc.expert_down(small._span(0, int(ids[t, j])), wl.H, wl.I,
                                                   hq[t * wl.k + j]) for j in range(wl.k))
        assert rel_l2(got[t], ref) <= 1e-5, t


def _forward_and_h(setup, x, T):
    """forward on the device, then the gate/up step on the forward's own ids
    (the same GEMM on the same inputs: the h the forward rounded)."""
    import torch
    wl = setup.wl
    xd = to_dev_bf16(x)
    out = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    setup.m.forward(xd, T, out, ids, w, out_f32=out32)
    hbuf = torch.empty((T * wl.k, wl.I), dtype=torch.float32, device="cuda")
    setup.m.step_expert_gateup(0, xd, T, ids, hbuf)
    setup.m.sync()
    return (out32.cpu().numpy(), out.cpu().numpy().view(np.uint16), ids.cpu().numpy(),
            w.cpu().numpy(), hbuf.cpu().numpy())


def h_in_oracle_order(ids, h, ref_ids):
    """The device's h rows (t*k + device slot) in the oracle's slot order,
    matched by expert id (two selected experts may sit in either order)."""
    T, k = ref_ids.shape
    out = np.empty_like(h)
    for t in range(T):
        for j in range(k):
            jj = int(np.nonzero(ids[t] == ref_ids[t, j])[0][0])
            out[t * k + j] = h[t * k + jj]
    return out


def mxfp8_reference(layer, x, ids, h):
    """The oracle's MXFP8 layer on the device's h (ids checked first)."""
    o_ids, o_w = orc.topk_softmax(orc.router_logits(layer.router, x), layer.s.k)
    check_ids_weights(ids, np.ones(ids.shape), o_ids, np.ones(o_ids.shape))
    return orc.moe_layer_mxfp8(layer, x, h_in=h_in_oracle_order(ids, h, o_ids))


@pytest.mark.parametrize("T", [1, 5, 40])
def test_forward_small(small, torch, T):
    x = draw_tokens(small, T, first_id=500 + T)
    out32, out, ids, w, h = _forward_and_h(small, x, T)
    ref = mxfp8_reference(small.layers[0], x, ids, h)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])
    assert np.array_equal(out, np.array([[orc.f64_to_bf16(v) for v in row] for row in out32]))
    # against the exact layer: the two roundings (x and h, ~2-3 % each for
    # Gaussian blocks) leave a few per cent; never zero
    exact = orc.moe_layer(small.layers[0], x)
    d = rel_l2(out32, exact["out"])
    assert 1e-4 < d < 0.1, d


@pytest.fixture(scope="module")
def k3(torch):
    s = Setup(K3, max_tokens=512, mxfp8=True)
    yield s
    s.close()


def test_k3_decode_one_token(k3, torch):
    x = draw_tokens(k3, 1, first_id=900)
    out32, _, ids, w, h = _forward_and_h(k3, x, 1)
    ref = mxfp8_reference(k3.layers[0], x, ids, h)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


def test_k3_batch512_sampled(k3, torch):
    T = 512
    x = np.stack([synth.token(K3.seed, K3.cfg_id, 7000 + t, K3.H) for t in range(T)])
    out32, _, ids, w, h = _forward_and_h(k3, x, T)
    assert np.all(np.isfinite(out32))
    routers = k3.routers[0]
    sample = [0, 1, 77, 255, 256, 300, 444, 511]
    logits = orc.router_logits(routers, x[sample])
    o_ids, o_w = orc.topk_softmax(logits, K3.k)
    gaps = np.sort(logits, axis=1)[:, ::-1]
    for i, t in enumerate(sample):
        if gaps[i, K3.k - 1] - gaps[i, K3.k] < 1e-3:
            continue   # a near tie: either order is a correct selection
        check_ids_weights(ids[t:t + 1], w[t:t + 1], o_ids[i:i + 1], o_w[i:i + 1])
        ref = mxfp8_reference(k3.layers[0], x[t:t + 1], ids[t:t + 1],
                              h[t * K3.k:(t + 1) * K3.k])
        check_out(out32[t:t + 1], ref["out"])
