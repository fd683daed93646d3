"""The exact block-scaled batch path (DF_MOE_PLANES) against the oracle.

The routed experts run on the same block-scaled MXFP4 x E4M3 tensor-core
GEMMs as the MXFP8 variant, but every activation enters them as a sum of
E4M3 planes (x: 4, h: 5), each the MXFP8 rounding of what the planes before
it left, with its own block exponent. The remainder after the last plane is
below fp32 precision of the block for any bf16 x whose block spans up to
~2^40 (one outlier block included) and for fp32 h, so the path is held to the
exact path's bars against the exact oracle: single steps at 1e-5 relative L2
(fp32 sums of exact products), layer outputs at the layer bars, ids exact.
Shapes: a small layer (H = 256, I = 128, 8 experts, top-2) with a hot expert
taking several passes (16 tokens a pass), hidden
states at the edges of the range, and the K3 layer at batch 512.
"""
import numpy as np
import pytest

import oracle as orc
import synth
from synth.workloads import Workload
from moe_setup import (Setup, check_ids_weights, check_out, draw_tokens, range_tokens, rel_l2,
                       to_dev_bf16)

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
    s = Setup(SMALL, max_tokens=160, planes=True)
    yield s
    s.close()


def x_f64(x):
    return (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def _ids_hot(T, k, E, hot, seed):
    rng = np.random.default_rng(seed)
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        ids[t] = [hot] + [e for e in rng.permutation(E) if e != hot][:k - 1]
    return ids


@pytest.mark.parametrize("T", [1, 7, 100])
def test_gateup_step(small, torch, T):
    wl = SMALL
    x = np.stack([synth.token(wl.seed, wl.cfg_id, 700 + t, wl.H) for t in range(T)])
    ids = _ids_hot(T, wl.k, wl.E, hot=2, seed=T)   # expert 2: T tokens (7 passes at 100)
    hbuf = torch.zeros((T * wl.k, wl.I), dtype=torch.float32, device="cuda")
    small.m.step_expert_gateup(0, to_dev_bf16(x), T, torch.from_numpy(ids).cuda(), hbuf)
    torch.cuda.synchronize()
    got = hbuf.cpu().numpy().astype(np.float64)
    for t in range(T):
        for j in range(wl.k):
            ref = orc.expert_gateup(small._span(0, int(ids[t, j])), wl.H, wl.I, x_f64(x[t]))
            assert rel_l2(got[t * wl.k + j], ref) <= 1e-5, (t, j)


@pytest.mark.parametrize("T", [1, 13, 100])
def test_down_step(small, torch, T):
    wl = SMALL
    rng = np.random.default_rng(80 + T)
    h = (rng.standard_normal((T * wl.k, wl.I)) *
         np.ldexp(1.0, rng.integers(-6, 6, (T * wl.k, 1)))).astype(np.float32)
    h[0, 5] *= 2.0 ** 20                            # an outlier in one block
    ids = _ids_hot(T, wl.k, wl.E, hot=5, seed=200 + T)
    w = rng.uniform(0.1, 1.0, (T, wl.k)).astype(np.float32)
    y = torch.zeros((T, wl.H), dtype=torch.float32, device="cuda")
    small.m.step_expert_down(0, torch.from_numpy(h).cuda(), T, torch.from_numpy(ids).cuda(),
                             torch.from_numpy(w).cuda(), y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    for t in range(T):
        ref = sum(float(w[t, j]) * orc.expert_down(small._span(0, int(ids[t, j])), wl.H, wl.I,
                                                   h[t * wl.k + j].astype(np.float64))
                  for j in range(wl.k))
        assert rel_l2(got[t], ref) <= 1e-5, t


def _forward(m, x, T, torch):
    wl_H = x.shape[1]
    out = torch.empty((T, wl_H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, wl_H), dtype=torch.float32, device="cuda")
    k = m.cfg.top_k
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32)
    m.sync()
    return out.cpu().numpy().view(np.uint16), out32.cpu().numpy(), ids.cpu().numpy(), \
        w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 5, 40])
def test_forward_small(small, torch, T):
    x = draw_tokens(small, T, first_id=900 + T)
    out, out32, ids, w = _forward(small.m, x, T, torch)
    ref = orc.moe_layer(small.layers[0], x)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])
    rne = torch.from_numpy(out32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, rne)


def test_input_range(small, torch):
    """Tokens scaled by 2^20 and 2^-60, and one with a 2^20 and a 2^-40
    chunk: every block carries its own exponents, plane by plane."""
    xs = range_tokens(small, first_id=31000)
    out, out32, ids, w = _forward(small.m, xs, 3, torch)
    assert np.all(np.isfinite(out32))
    ref = orc.moe_layer(small.layers[0], xs)
    check_ids_weights(ids, w, ref["ids"], ref["w"])
    check_out(out32, ref["out"])


@pytest.mark.parametrize("T", [5, 40, 100])
def test_forward_equals_steps(small, torch, T):
    """The forward splits x once per token and copies the planes to every
    assignment's rows; the gate/up step does the same from the caller's x,
    and the down step splits the h it is given as the forward splits its
    own. So the forward's output equals, bit for bit, the steps' routed sum
    plus the shared part (added in fp32, as the forward adds them)."""
    wl = SMALL
    x = draw_tokens(small, T, first_id=1200 + T)
    _, out32, ids, w = _forward(small.m, x, T, torch)
    xd = to_dev_bf16(x)
    idd = torch.from_numpy(ids).cuda()
    wd = torch.from_numpy(w).cuda()
    hbuf = torch.empty((T * wl.k, wl.I), dtype=torch.float32, device="cuda")
    small.m.step_expert_gateup(0, xd, T, idd, hbuf)
    y = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
    small.m.step_expert_down(0, hbuf, T, idd, wd, y)
    ysh = torch.empty((T, wl.H), dtype=torch.float32, device="cuda")
    small.m.step_shared(0, xd, T, ysh)
    small.m.sync()
    want = y.cpu().numpy() + ysh.cpu().numpy()
    assert want.dtype == np.float32
    assert np.array_equal(out32.view(np.uint32), want.view(np.uint32))


@pytest.fixture(scope="module")
def k3(torch):
    s = Setup(K3, max_tokens=512, planes=True)
    yield s
    s.close()


def test_k3_batch512(k3, torch):
    T = 512
    x = np.stack([synth.token(K3.seed, K3.cfg_id, 9000 + t, K3.H) for t in range(T)])
    out, out32, ids, w = _forward(k3.m, x, T, torch)
    rid, rw = orc.topk_softmax(orc.router_logits(k3.routers[0], x), K3.k)
    logits = orc.router_logits(k3.routers[0], x)
    srt = np.sort(logits, axis=1)[:, ::-1]
    clear = srt[:, K3.k - 1] - srt[:, K3.k] >= 1e-3   # tokens without a near tie
    check_ids_weights(ids[clear], w[clear], rid[clear], rw[clear])
    sample = [t for t in list(range(0, T, 32)) + [T - 1] if clear[t]]
    ref = orc.moe_layer(k3.layers[0], x[sample])
    check_out(out32[sample], ref["out"])
    assert np.all(np.isfinite(out32))


def test_k3_decode_batch1(k3, torch):
    """One token on a planes handle runs the two phase kernels with the
    routed experts on the block-scaled MMA (gate/up in eight parts of K, h =
    SwiGLU of the parts' sums): full outputs at the layer bars, ids exact."""
    for t in range(3):
        x = np.stack([synth.token(K3.seed, K3.cfg_id, 9700 + t, K3.H)])
        out, out32, ids, w = _forward(k3.m, x, 1, torch)
        ref = orc.moe_layer(k3.layers[0], x)
        check_ids_weights(ids, w, ref["ids"], ref["w"])
        check_out(out32, ref["out"])
        rne = torch.from_numpy(out32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(out, rne)


def test_k3_decode_batch1_repeatable(k3, torch):
    """The phase path's sums run in a fixed order: the same token twice gives
    the same bits."""
    x = np.stack([synth.token(K3.seed, K3.cfg_id, 9750, K3.H)])
    a = _forward(k3.m, x, 1, torch)[1]
    b = _forward(k3.m, x, 1, torch)[1]
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


# no shared experts (every CTA of the phase kernels routed), and a K that
# the eight parts split unevenly (H = 1280: 10 stages of 128, parts of one
# and two stages)
NOSH = Workload("noshared-h1280-i384-e12-top3", 6, H=1280, I=384, E=12, k=3, n_shared=0,
                Is=0, T=1)


@pytest.mark.parametrize("wl", [NOSH])
def test_decode_batch1_shapes(wl, torch):
    s = Setup(wl, max_tokens=4, planes=True)
    try:
        for t in range(2):
            x = draw_tokens(s, 1, first_id=4100 + t)
            out, out32, ids, w = _forward(s.m, x, 1, torch)
            ref = orc.moe_layer(s.layers[0], x)
            check_ids_weights(ids, w, ref["ids"], ref["w"])
            check_out(out32, ref["out"])
    finally:
        s.close()
