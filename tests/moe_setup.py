"""Shared set-up of the tests: handles loaded with a workload's synthetic
weights, tokens drawn with the routing-gap rule, and the parity checks.

The gap rule (expert ids must match exactly, so a token whose k-th and
(k+1)-th oracle logits are closer than 1e-3 at any layer is redrawn from the
next sub-seed) uses the oracle's own logits.
"""
import numpy as np

import oracle as orc
import synth

GAP = 1e-3


def torch_mod():
    import torch
    return torch


def to_dev_bf16(a):
    """numpy uint16 bf16 bits -> int16 device tensor (same bits)."""
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(
        np.float32).astype(np.float64)


def layer_weights(wl, layer):
    router = synth.router(wl.seed, wl.wcfg, layer, wl.E, wl.H)
    shared = [synth.shared(wl.seed, wl.wcfg, layer, s, wl.H, wl.Is)
              for s in range(wl.n_shared)]
    return router, shared


class Setup:
    """A df_moe handle with every layer of workload `wl` loaded, plus the
    oracle's view of the same weights (spans generated on demand on the
    host)."""

    def __init__(self, wl, max_tokens=None, chunk=64, mma_sync_prefill=False,
                 cache_slots=0, mxfp8=False, planes=False):
        import mxfp4_routed_expert_top_gb300 as dfm
        torch = torch_mod()
        self.wl = wl
        flags = ((dfm.STACK_RMSNORM_RESIDUAL if wl.stack else 0)
                 | (dfm.PREFILL_MMA_SYNC if mma_sync_prefill else 0)
                 | (dfm.MXFP8_ACT if mxfp8 else 0)
                 | (dfm.PLANES if planes else 0))
        self.m = dfm.MoE(wl.H, wl.E, wl.k, wl.I, wl.n_shared, wl.Is,
                         n_layers=wl.L, max_tokens=max_tokens or wl.T,
                         rms_eps=wl.eps, flags=flags, cache_slots=cache_slots)
        self.routers, self.shared, self.layers = [], [], []
        span = synth.span_bytes(wl.H, wl.I)
        stream = torch.cuda.current_stream()
        buf = torch.empty(min(chunk, wl.E) * span, dtype=torch.uint8, device="cuda")
        for l in range(wl.L):
            router, shared = layer_weights(wl, l)
            self.routers.append(router)
            self.shared.append(shared)
            self.m.load_experts(l, router=router, shared=shared)
            for e0 in range(0, wl.E, chunk):
                n = min(chunk, wl.E - e0)
                synth.dev_expert_spans(wl.seed, wl.wcfg, l, e0, n, wl.H, wl.I,
                                       buf.data_ptr(), stream.cuda_stream)
                self.m.load_experts(l, experts=buf, expert_begin=e0, expert_count=n,
                                    src_is_device=True, stream=stream)
            self.layers.append(orc.Layer(wl.H, wl.E, wl.k, wl.I, wl.Is, router, shared,
                                         self._span, layer=l))
        torch.cuda.synchronize()
        del buf
        self._cache = {}

    def _span(self, layer, e):
        return synth.expert_spans(self.wl.seed, self.wl.wcfg, layer, e, 1,
                                  self.wl.H, self.wl.I)[0]

    def close(self):
        self.m.close()
        for L in self.layers:
            L.clear_cache()


def gap_ok(logits, k):
    """True when the k-th and (k+1)-th largest logits differ by >= GAP."""
    if k >= logits.shape[-1]:
        return True
    s = np.sort(logits, axis=-1)[..., ::-1]
    return bool(np.all(s[..., k - 1] - s[..., k] >= GAP))


def draw_tokens(setup, T, first_id=0):
    """T tokens of the workload's cfg stream that pass the gap rule at the
    first layer (single-layer workloads)."""
    wl = setup.wl
    out = []
    for t in range(T):
        for r in range(synth.gen.REDRAWS_PER_TOKEN):
            x = synth.token(wl.seed, wl.cfg_id, first_id + t, wl.H, redraw=r)
            if gap_ok(orc.router_logits(setup.routers[0], x), wl.k):
                out.append(x)
                break
        else:
            raise RuntimeError("no token passed the gap rule")
    return np.stack(out)


def scaled_bits(x, p):
    """bf16 bits of x * 2^p (exact: a power of two, no overflow or underflow)."""
    f = (np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    y = f * np.float32(2.0 ** p)
    assert np.all(np.isfinite(y)) and np.all((y == 0) == (f == 0))
    return (y.view(np.uint32) >> 16).astype(np.uint16)


def range_tokens(setup, first_id, chunk=512):
    """Three tokens at the edges of the hidden state's range: one scaled by
    2^20 (~1e6), one by 2^-60 (~1e-18), and one whose first 512-column chunk
    is scaled by 2^20 and second by 2^-40 (the rest N(0,1)). Scaling a token
    by a power of two scales its logits exactly, so tokens that passed the
    gap rule still pass it; the mixed token is checked on its own."""
    wl = setup.wl
    base = draw_tokens(setup, 2, first_id=first_id)
    big, small = scaled_bits(base[0], 20), scaled_bits(base[1], -60)
    for r in range(synth.gen.REDRAWS_PER_TOKEN):
        x = synth.token(wl.seed, wl.cfg_id, first_id + 2, wl.H, redraw=r)
        mixed = x.copy()
        c1 = min(chunk, wl.H // 2)
        mixed[:c1] = scaled_bits(x[:c1], 20)
        mixed[c1:2 * c1] = scaled_bits(x[c1:2 * c1], -40)
        if gap_ok(orc.router_logits(setup.routers[0], mixed), wl.k):
            return np.stack([big, small, mixed])
    raise RuntimeError("no mixed token passed the gap rule")


def draw_stack_token(setup, token_id):
    """One token for a stack workload that passes the gap rule at every
    layer; returns (x, oracle result of the stack for it)."""
    wl = setup.wl
    for r in range(synth.gen.REDRAWS_PER_TOKEN):
        x = synth.token(wl.seed, wl.cfg_id, token_id, wl.H, redraw=r)[None, :]
        ref = orc.moe_stack(setup.layers, x, wl.eps)
        if gap_ok(ref["logits"], wl.k):
            return x[0], ref
    raise RuntimeError("no token passed the gap rule")


def check_ids_weights(got_ids, got_w, ref_ids, ref_w, wtol=1e-5):
    """Ids as sets per token (bit exact); weights keyed by id."""
    got_ids = np.asarray(got_ids).reshape(-1, ref_ids.shape[-1])
    got_w = np.asarray(got_w).reshape(got_ids.shape)
    ref_ids = ref_ids.reshape(got_ids.shape)
    ref_w = ref_w.reshape(got_ids.shape)
    for t in range(got_ids.shape[0]):
        assert sorted(got_ids[t].tolist()) == sorted(ref_ids[t].tolist()), \
            "token %d: ids %s vs oracle %s" % (t, got_ids[t], ref_ids[t])
        gw = dict(zip(got_ids[t].tolist(), got_w[t].tolist()))
        for e, w in zip(ref_ids[t].tolist(), ref_w[t].tolist()):
            assert abs(gw[e] - w) <= wtol, "token %d expert %d: w %r vs %r" % (t, e, gw[e], w)


def check_out(got, ref, rel_l2=2e-3, max_abs_rms=1e-2):
    """Layer output tolerance: relative L2 <= 2e-3 and max-abs error <=
    1e-2 x RMS of the oracle output (per token)."""
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    for t in range(ref.shape[0]):
        r, g = ref[t], got[t]
        rms = np.sqrt(np.mean(r ** 2))
        rel = np.linalg.norm(g - r) / np.linalg.norm(r)
        mx = np.max(np.abs(g - r))
        assert rel <= rel_l2, "token %d: relative L2 %.3e" % (t, rel)
        assert mx <= max_abs_rms * rms, "token %d: max abs %.3e vs rms %.3e" % (t, mx, rms)


def rel_l2(got, ref):
    got = np.asarray(got, dtype=np.float64).reshape(ref.shape)
    return np.linalg.norm(got - ref) / np.linalg.norm(ref)
