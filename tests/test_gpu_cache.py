"""GPU parity of the expert cache: every expert in pinned host memory, a few
slots of them a layer in HBM, filled on demand (the Deltafin README's
previous-token reuse and the kimi-k3-in-c blog's expert LRU cache, moved from
SSD -> RAM to Grace memory -> HBM).

Outputs must equal the oracle's under the layer tolerance whatever the
cache holds. The policy (a selected expert not cached takes an empty slot,
else the least recently used slot not needed by this call, the lowest such
slot on equal use) is pinned by a host model of it fed with the oracle's
selections: hits, misses and bytes copied must match it exactly. Bytes, not
hits, are the measure that counts (the blog's first trap).
"""
import numpy as np
import pytest

import oracle as orc
import synth
from moe_setup import (Setup, bits_to_f64, check_ids_weights, check_out, draw_tokens,
                       to_dev_bf16)

pytestmark = pytest.mark.gpu

TINY, K3 = synth.WORKLOADS[0], synth.WORKLOADS[1]


@pytest.fixture(scope="module")
def torch():
    import torch as t
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    return t


class LruModel:
    """Host model of the cache policy, one layer."""

    def __init__(self, slots):
        self.expert_of = [-1] * slots
        self.used = [0] * slots
        self.slot_of = {}
        self.clock = 0
        self.hits = self.misses = 0

    def call(self, ids):
        self.clock += 1
        now = self.clock
        miss = []
        for e in ids:
            sl = self.slot_of.get(e)
            if sl is not None:
                if self.used[sl] != now:
                    self.used[sl] = now
                    self.hits += 1
            elif e not in miss:
                miss.append(e)
        for e in miss:
            v = -1
            for sl in range(len(self.used)):
                if self.used[sl] == now:
                    continue
                if self.expert_of[sl] < 0:
                    v = sl
                    break
                if v < 0 or self.used[sl] < self.used[v]:
                    v = sl
            assert v >= 0
            if self.expert_of[v] >= 0:
                del self.slot_of[self.expert_of[v]]
            self.expert_of[v] = e
            self.slot_of[e] = v
            self.used[v] = now
            self.misses += 1


def _forward(m, x, T, torch, H, k):
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    out32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    m.forward(to_dev_bf16(x), T, out, ids, w, out_f32=out32)
    m.sync()
    return out32.cpu().double().numpy(), ids.cpu().numpy(), w.cpu().double().numpy()


def test_lru_model_pins():
    """The host model itself against hand-worked sequences (2 slots)."""
    m = LruModel(2)
    m.call([5, 3])                      # both miss: 5 -> slot 0, 3 -> slot 1
    assert (m.hits, m.misses, m.expert_of) == (0, 2, [5, 3])
    m.call([3, 3])                      # one distinct hit
    assert (m.hits, m.misses) == (1, 2)
    m.call([7])                         # evicts 5 (slot 0, used at call 1)
    assert (m.hits, m.misses, m.expert_of) == (1, 3, [7, 3])
    m.call([3, 5])                      # 3 hits; 5 evicts 7 (call 3) not 3 (now)
    assert (m.hits, m.misses, m.expert_of) == (2, 4, [5, 3])


@pytest.fixture(scope="module")
def tiny_cached(torch):
    s = Setup(TINY, max_tokens=2, cache_slots=5)
    yield s
    s.close()


def test_tiny_cached_matches_oracle_and_policy(tiny_cached, torch):
    s, wl = tiny_cached, TINY
    span = s.m.span_bytes
    model = LruModel(5)
    x = draw_tokens(s, 24, first_id=500)
    calls = [x[t:t + 1] for t in range(12)] + [x[t:t + 2] for t in range(12, 24, 2)]
    calls += [x[3:4], x[3:4], x[12:14]]  # repeats: every expert found cached
    for xc in calls:
        T = xc.shape[0]
        h0, m0, _ = s.m.cache_stats()
        out32, ids, w = _forward(s.m, xc, T, torch, wl.H, wl.k)
        ref = orc.moe_layer(s.layers[0], xc)
        check_ids_weights(ids, w, ref["ids"], ref["w"])
        check_out(out32, ref["out"])
        model.call(ref["ids"].reshape(-1).tolist())
        hits, misses, nbytes = s.m.cache_stats()
        assert (hits, misses) == (model.hits, model.misses)
        assert nbytes == misses * span
        assert hits - h0 + misses - m0 == len(set(ref["ids"].reshape(-1).tolist()))
    # the last three calls repeat earlier selections still cached
    assert model.misses < len(calls) * wl.k


def test_tiny_cached_reload_and_readback(tiny_cached, torch):
    """A reloaded expert leaves the cache; the read-back gives the canonical
    span from the host pool."""
    s, wl = tiny_cached, TINY
    x = draw_tokens(s, 1, first_id=700)
    ref = orc.moe_layer(s.layers[0], x)
    _forward(s.m, x, 1, torch, wl.H, wl.k)
    h0, m0, _ = s.m.cache_stats()
    _forward(s.m, x, 1, torch, wl.H, wl.k)
    h1, m1, _ = s.m.cache_stats()
    assert (h1 - h0, m1 - m0) == (wl.k, 0)
    e = int(ref["ids"][0, 0])
    spans = synth.expert_spans(wl.seed, wl.wcfg, 0, e, 1, wl.H, wl.I)
    s.m.load_experts(0, experts=spans, expert_begin=e, expert_count=1)
    out32, ids, w = _forward(s.m, x, 1, torch, wl.H, wl.k)
    h2, m2, _ = s.m.cache_stats()
    assert (h2 - h1, m2 - m1) == (wl.k - 1, 1)
    check_out(out32, ref["out"])
    got = np.empty(s.m.span_bytes, dtype=np.uint8)
    s.m.read_expert_span(0, e, got)
    assert np.array_equal(got, spans[0])


def test_cache_guards(tiny_cached, torch):
    import mxfp4_routed_expert_top_gb300 as dfm
    wl = TINY
    for kw in (dict(max_tokens=2, cache_slots=3),      # < max_tokens * top_k
               dict(max_tokens=1, cache_slots=9),      # > n_experts
               dict(max_tokens=16, cache_slots=8),     # beyond decode batches
               dict(max_tokens=1, cache_slots=4, flags=2)):  # a reserved flag bit
        with pytest.raises(dfm.DfMoeError) as ei:
            dfm.MoE(wl.H, wl.E, wl.k, wl.I, wl.n_shared, wl.Is, **kw)
        assert ei.value.code == -1
    s = tiny_cached
    x = to_dev_bf16(draw_tokens(s, 1, first_id=800))
    out = torch.empty((1, wl.H), dtype=torch.int16, device="cuda")
    ids = torch.empty((1, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, wl.k), dtype=torch.float32, device="cuda")
    with pytest.raises(dfm.DfMoeError) as ei:
        s.m.graph(x, 1, out, ids, w)
    assert ei.value.code == -1
    hbuf = torch.empty((1, 2 * wl.I), dtype=torch.float32, device="cuda")
    with pytest.raises(dfm.DfMoeError) as ei:
        s.m.step_expert_gateup(0, x, 1, ids, hbuf)
    assert ei.value.code == -1
    with dfm.MoE(wl.H, wl.E, wl.k, wl.I, wl.n_shared, wl.Is) as plain:
        assert plain.cache_stats() == (0, 0, 0)


@pytest.fixture(scope="module")
def k3_cached(torch):
    s = Setup(K3, max_tokens=2, cache_slots=40)
    yield s
    s.close()
    torch.cuda.empty_cache()


def test_k3_cached_matches_oracle(k3_cached, torch):
    """K3 layer (896 experts, 15.7 GB in pinned host memory) through 40 HBM
    slots: three tokens, a repeat, then a batch of two."""
    s, wl = k3_cached, K3
    span = s.m.span_bytes
    model = LruModel(40)
    x = draw_tokens(s, 4, first_id=40)
    calls = [x[0:1], x[1:2], x[2:3], x[2:3], x[0:2], x[3:4]]
    for i, xc in enumerate(calls):
        T = xc.shape[0]
        out32, ids, w = _forward(s.m, xc, T, torch, wl.H, wl.k)
        ref = orc.moe_layer(s.layers[0], xc)
        check_ids_weights(ids, w, ref["ids"], ref["w"])
        check_out(out32, ref["out"])
        model.call(ref["ids"].reshape(-1).tolist())
        hits, misses, nbytes = s.m.cache_stats()
        assert (hits, misses) == (model.hits, model.misses), "call %d" % i
        assert nbytes == misses * span
    # the repeated token moved no bytes
    assert model.hits >= wl.k


@pytest.fixture(scope="module")
def k3_cached8(torch):
    s = Setup(K3, max_tokens=8, cache_slots=128)
    yield s
    s.close()
    torch.cuda.empty_cache()


def test_k3_cached_batch8(k3_cached8, torch):
    """Batches of 8 tokens (up to 128 distinct experts a call) through 128
    slots: the second batch evicts most of the first; the third repeats
    the first and must find only what the second left."""
    s, wl = k3_cached8, K3
    span = s.m.span_bytes
    model = LruModel(128)
    x = draw_tokens(s, 16, first_id=300)
    for i, xc in enumerate([x[0:8], x[8:16], x[0:8], x[4:8]]):
        T = xc.shape[0]
        out32, ids, w = _forward(s.m, xc, T, torch, wl.H, wl.k)
        ref = orc.moe_layer(s.layers[0], xc)
        check_ids_weights(ids, w, ref["ids"], ref["w"])
        check_out(out32, ref["out"])
        model.call(ref["ids"].reshape(-1).tolist())
        hits, misses, nbytes = s.m.cache_stats()
        assert (hits, misses) == (model.hits, model.misses), "call %d" % i
        assert nbytes == misses * span


def test_tiny_stack_cached(torch):
    """Three tiny layers with RMSNorm and residual, each with its own 3 HBM
    slots: bit-identical to the resident handle (same kernels on the same
    span bytes), and every layer against the oracle on the inputs the device
    gave it."""
    import dataclasses
    from moe_setup import gap_ok
    wl = dataclasses.replace(TINY, name="tiny-stack3", L=3, stack=True)
    cached = Setup(wl, max_tokens=2, cache_slots=4)
    resident = Setup(wl, max_tokens=2)
    try:
        L, H, k = wl.L, wl.H, wl.k
        for T, first in ((1, 40), (2, 60), (1, 40)):
            res = {}
            for name, s in (("cached", cached), ("resident", resident)):
                out = torch.empty((T, H), dtype=torch.int16, device="cuda")
                out32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
                ids = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
                w = torch.empty((L, T, k), dtype=torch.float32, device="cuda")
                tx = torch.empty((L, T, H), dtype=torch.int16, device="cuda")
                txn = torch.empty((L, T, H), dtype=torch.int16, device="cuda")
                x = np.stack([synth.token(wl.seed, wl.cfg_id, first + t, H) for t in range(T)])
                s.m.forward_trace(to_dev_bf16(x), T, out, ids, w, trace_x=tx, trace_xn=txn,
                                  out_f32=out32)
                s.m.sync()
                res[name] = [a.cpu().numpy() for a in (out, out32, ids, w, tx, txn)]
            for a, b in zip(res["cached"], res["resident"]):
                assert np.array_equal(a, b)
            out, out32, ids, w, tx, txn = res["cached"]
            tx, txn = tx.view(np.uint16), txn.view(np.uint16)
            for l in range(L):
                if not all(gap_ok(orc.router_logits(cached.routers[l], txn[l, t:t + 1]), k)
                           for t in range(T)):
                    continue  # ids of a near-tie are not unique
                ref = orc.moe_layer(cached.layers[l], txn[l], residual=tx[l])
                check_ids_weights(ids[l], w[l], ref["ids"], ref["w"])
                y_ref = ref["out"] - bits_to_f64(tx[l])
                if l == L - 1:
                    check_out(out32 - bits_to_f64(tx[l]), y_ref)
                else:
                    # the next input is the bf16 rounding of residual + output:
                    # within one ulp of the oracle sum's rounding (plus 1e-3 x
                    # RMS of the output where the two nearly cancel)
                    want = np.array([[orc.f64_to_bf16(v) for v in row] for row in ref["out"]],
                                    dtype=np.uint16)
                    slack = 1e-3 * np.sqrt(np.mean(y_ref ** 2, axis=-1, keepdims=True))
                    ulp = np.abs(bits_to_f64(want)) * 2.0 ** -7
                    diff = np.abs(bits_to_f64(tx[l + 1]) - bits_to_f64(want))
                    assert np.all(diff <= ulp + slack), "layer %d" % l
        hits, misses, _ = cached.m.cache_stats()
        assert misses >= k * L and hits + misses >= 3 * k * L
    finally:
        cached.close()
        resident.close()
