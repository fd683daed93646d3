"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against what the pages print, a closed
form, ml_dtypes (the Deltafin README's own e2m1 bit-exactness reference,
"Thanks"), a library routine (numpy matmul / sort, scipy, torch casts) or
brute force on tiny inputs — chosen so that a plausible slip (swapped nibble
order, wrong scale index, gate/up swapped, transposed down matrix, dropped
shared term, wrong softmax base, unstable tie order) fails at least one.
No CUDA here.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as orc
import synth

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "k3_pages_arithmetic.json")))
K3H, K3I = 7168, 1536


def g(name):
    return GOLD[name]["value"]


# ---- independent helpers (written from the format definitions, not the oracle)

def e2m1_from_fields(code):
    """OCP E2M1: sign bit 3, 2-bit exponent (bias 1), 1-bit mantissa;
    exponent 0 is subnormal (0.5 * m)."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    return s * (0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m))


def unpack_codes(q):
    """[rows, cols/2] packed bytes -> [rows, cols] codes, low nibble first."""
    lo = q & 0x0F
    hi = q >> 4
    out = np.empty((q.shape[0], q.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def dequant_ml_dtypes(q, s):
    ml = pytest.importorskip("ml_dtypes")
    codes = unpack_codes(q)
    vals = codes.view(ml.float4_e2m1fn).astype(np.float64)
    scale = np.ldexp(1.0, s.astype(np.int64) - 127)
    return vals * np.repeat(scale, 32, axis=1)


def bf16_bits_to_f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(
        np.float32).astype(np.float64)


def split_span(span, H, I):
    """Slice a canonical span by the documented layout (independently of the
    oracle's own offsets)."""
    q, s = H * I // 2, H * I // 32
    sizes = [q, s, q, s, q, s]
    shapes = [(I, H // 2), (I, H // 32), (I, H // 2), (I, H // 32),
              (H, I // 2), (H, I // 32)]
    out, o = [], 0
    for n, sh in zip(sizes, shapes):
        out.append(span[o:o + n].reshape(sh))
        o += n
    assert o == span.size
    return out


def ffn_numpy(span, H, I, x):
    gq, gs, uq, us, dq, ds = split_span(span, H, I)
    G, U, D = dequant_ml_dtypes(gq, gs), dequant_ml_dtypes(uq, us), dequant_ml_dtypes(dq, ds)
    gx, ux = G @ x, U @ x
    h = gx / (1.0 + np.exp(-gx)) * ux
    return D @ h


def shared_numpy(gate, up, down, x):
    G, U, D = bf16_bits_to_f64(gate), bf16_bits_to_f64(up), bf16_bits_to_f64(down)
    gx, ux = G @ x, U @ x
    return D @ (gx / (1.0 + np.exp(-gx)) * ux)


# ---- the pages' printed arithmetic ------------------------------------------

def test_span_bytes_match_pages():
    assert orc.span_bytes(K3H, K3I) == g("expert_span_bytes")
    assert orc.span_bytes(K3H, K3I) / (3 * K3H * K3I) == g("bytes_per_weight")
    # 4 bits of value + 8 bits of exponent per block of 32
    assert 0.5 + 1.0 / g("block_elements") == g("bytes_per_weight")


def test_intermediate_size_follows_from_pages():
    inter = g("expert_span_bytes") / g("bytes_per_weight") / 3 / g("hidden")
    assert inter == K3I


def test_expert_pool_and_per_token_bytes():
    total = g("routed_experts_total") * g("expert_span_bytes")
    assert g("routed_experts_total") == g("moe_layers") * g("experts_per_layer")
    # the page prints 1.447 TB for 1,446,456,066,048 B (it rounds the last
    # digit up); agreement to the printed precision is what can be checked
    assert abs(total / 1e12 - g("experts_total_tb")) <= 1e-3
    assert round(100 * total / g("checkpoint_bytes")) == g("experts_share_of_checkpoint_pct")
    per_token = g("top_k") * g("moe_layers") * orc.span_bytes(K3H, K3I)
    assert round(per_token / 1e9, 2) == g("expert_gb_per_token_blog")
    assert abs(g("top_k") * g("moe_layers") * g("expert_mb") -
               g("expert_mb_per_token_analysis")) < 1e-6
    assert round(g("expert_span_bytes") / 1e6, 2) == g("expert_mb")
    assert round(100 * g("top_k") / g("experts_per_layer"), 2) == g("touched_fraction_pct")


def test_span_offsets_are_six_contiguous_tensors():
    off = orc.span_offsets(K3H, K3I)
    sizes = np.diff(off + [orc.span_bytes(K3H, K3I)])
    q, s = K3H * K3I // 2, K3H * K3I // 32
    assert list(sizes) == [q, s, q, s, q, s]
    assert off[0] == 0


# ---- element formats ---------------------------------------------------------

def test_e2m1_table_matches_ml_dtypes_and_fields():
    ml = pytest.importorskip("ml_dtypes")
    codes = np.arange(16, dtype=np.uint8)
    ref = codes.view(ml.float4_e2m1fn).astype(np.float64)
    for c in range(16):
        v = orc.e2m1_value(c)
        assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c])
        assert v == e2m1_from_fields(c)


def test_e2m1_fields_without_ml_dtypes():
    for c in range(16):
        assert orc.e2m1_value(c) == e2m1_from_fields(c)
    assert sorted({abs(orc.e2m1_value(c)) for c in range(16)}) == \
        [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e8m0_all_exponents():
    for e in range(255):
        assert orc.e8m0_value(e) == math.ldexp(1.0, e - 127)
    assert math.isnan(orc.e8m0_value(255))


def test_dequantised_weights_exact_in_fp32_and_bf16():
    # every code x every scale the workload draws is exactly representable,
    # so fused and dequantise-then-multiply can agree bit for bit
    import torch
    for c in range(16):
        for e in range(119, 128):
            v = orc.e2m1_value(c) * orc.e8m0_value(e)
            assert float(np.float32(v)) == v
            assert torch.tensor(v, dtype=torch.float64).to(torch.bfloat16).double().item() == v


def test_bf16_widening_matches_torch():
    import torch
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 16, 4000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # drop inf/nan
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([orc.bf16_to_f64(b) for b in bits])
    assert np.array_equal(got, ref)


def test_bf16_rounding_ties_and_library():
    import torch
    # exact ties round to the even mantissa
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert orc.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    assert orc.f64_to_bf16(-(1.0 + 2.0 ** -8)) == 0xBF80
    assert orc.f64_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert orc.f64_to_bf16(0.0) == 0 and orc.f64_to_bf16(-0.0) == 0x8000
    rng = np.random.default_rng(2)
    v = rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f64_to_bf16(x) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---- MXFP4 matrices ----------------------------------------------------------

def test_single_nonzero_code_isolates_one_weight():
    rows, cols = 4, 128
    for (r, c, code) in [(0, 0, 1), (1, 1, 7), (2, 63, 9), (3, 64, 15), (3, 127, 4)]:
        q = np.zeros((rows, cols // 2), dtype=np.uint8)
        s = np.full((rows, cols // 32), 127, dtype=np.uint8)
        s[r, c // 32] = 120 + (c // 32)  # a distinct scale in the element's block
        q[r, c // 2] = code if c % 2 == 0 else code << 4
        W = orc.mx_dequant(q, s)
        nz = np.argwhere(W != 0)
        assert nz.tolist() == [[r, c]]
        assert W[r, c] == e2m1_from_fields(code) * 2.0 ** (120 + c // 32 - 127)


def test_dequant_matches_ml_dtypes_on_random_matrix():
    rng = np.random.default_rng(3)
    q = rng.integers(0, 256, (48, 96), dtype=np.uint8)
    s = rng.integers(119, 128, (48, 6), dtype=np.uint8)
    assert np.array_equal(orc.mx_dequant(q, s), dequant_ml_dtypes(q, s))


def test_fused_gemv_equals_dequantise_then_dense():
    # the Deltafin README's fused kernel "matches the reference bit-for-bit"
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, (96, 512), dtype=np.uint8)
    s = rng.integers(119, 128, (96, 32), dtype=np.uint8)
    x = rng.standard_normal(1024)
    y = orc.mx_gemv(q, s, x)
    ref = dequant_ml_dtypes(q, s) @ x
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # and against an explicit sequential sum over the dequantised row
    W = orc.mx_dequant(q, s)
    for r in (0, 17, 95):
        acc = 0.0
        for c in range(1024):
            acc += W[r, c] * x[c]
        assert y[r] == acc


# ---- router / top-k -----------------------------------------------------------

def test_router_logits_match_numpy():
    rng = np.random.default_rng(5)
    E, H, T = 24, 256, 3
    Wr = rng.standard_normal((E, H)).astype(np.float32)
    x = synth.normal_bf16(synth.key(9, 0, 0, 5, 0), T * H, 1.0).reshape(T, H)
    got = orc.router_logits(Wr, x)
    ref = bf16_bits_to_f64(x) @ Wr.astype(np.float64).T
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_topk_against_full_sort_and_brute_force():
    rng = np.random.default_rng(6)
    T, E, k = 50, 40, 7
    logits = rng.standard_normal((T, E))
    logits[0, :] = 1.0                    # all tied: lowest ids win, in order
    logits[1, [3, 9, 20]] = 5.0           # a tie at the top
    ids, w = orc.topk_softmax(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))  # brute force
        assert list(ids[t]) == order[:k]
        sel = logits[t, order[:k]]
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        assert np.allclose(w[t], ref, rtol=1e-13, atol=0)
        assert abs(w[t].sum() - 1.0) < 1e-14
        # weight ratios are exp of logit differences
        assert np.allclose(w[t, 1:] / w[t, 0], np.exp(sel[1:] - sel[0]), rtol=1e-12)
    assert list(ids[0]) == list(range(k))
    assert list(ids[1][:3]) == [3, 9, 20]
    # np.argsort(stable) on negated logits gives the same selection
    ref_ids = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)


def test_topk_k_equals_e_is_dense_softmax():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((3, 9))
    ids, w = orc.topk_softmax(logits, 9)
    for t in range(3):
        full = np.exp(logits[t] - logits[t].max()); full /= full.sum()
        assert np.allclose(w[t], full[ids[t]], rtol=1e-13)


def test_silu_closed_form():
    scipy_special = pytest.importorskip("scipy.special")
    for v in [-50.0, -3.5, -1e-3, 0.0, 1e-3, 0.7, 12.0, 80.0]:
        assert orc.silu(v) == pytest.approx(v * scipy_special.expit(v), rel=1e-14, abs=1e-300)
    assert orc.silu(0.0) == 0.0


# ---- experts -------------------------------------------------------------------

@pytest.fixture(scope="module")
def tiny_spans():
    return synth.expert_spans(0, 0, 0, 0, 8, 256, 64)


def test_expert_ffn_matches_numpy_dense(tiny_spans):
    H, I = 256, 64
    x = bf16_bits_to_f64(synth.token(0, 0, 0, H))
    for e in range(8):
        got = orc.expert_ffn(tiny_spans[e], H, I, x)
        ref = ffn_numpy(tiny_spans[e], H, I, x)
        assert np.allclose(got, ref, rtol=1e-11, atol=1e-9 * np.abs(ref).max())


def test_expert_gateup_and_down_steps(tiny_spans):
    H, I = 256, 64
    x = bf16_bits_to_f64(synth.token(0, 0, 1, H))
    gq, gs, uq, us, dq, ds = split_span(tiny_spans[3], H, I)
    G, U, D = dequant_ml_dtypes(gq, gs), dequant_ml_dtypes(uq, us), dequant_ml_dtypes(dq, ds)
    h = orc.expert_gateup(tiny_spans[3], H, I, x)
    gx, ux = G @ x, U @ x
    assert np.allclose(h, gx / (1 + np.exp(-gx)) * ux, rtol=1e-11, atol=1e-9)
    # gate and up are not interchangeable: the swapped form differs
    assert not np.allclose(h, ux / (1 + np.exp(-ux)) * gx)
    y = orc.expert_down(tiny_spans[3], H, I, h)
    assert np.allclose(y, D @ h, rtol=1e-11, atol=1e-9 * np.abs(D @ h).max())


def test_one_k3_expert_matches_numpy_dense():
    H, I = K3H, K3I
    span = synth.expert_spans(0, 1, 0, 123, 1, H, I)[0]
    x = bf16_bits_to_f64(synth.token(0, 1, 0, H))
    got = orc.expert_ffn(span, H, I, x)
    ref = ffn_numpy(span, H, I, x)
    assert np.allclose(got, ref, rtol=1e-10, atol=1e-10 * np.abs(ref).max())


def test_shared_ffn_matches_numpy():
    H, Is = 256, 64
    gt, up, dn = synth.shared(0, 0, 0, 0, H, Is)
    x = bf16_bits_to_f64(synth.token(0, 0, 0, H))
    got = orc.shared_ffn(gt, up, dn, x)
    ref = shared_numpy(gt, up, dn, x)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


# ---- grouping --------------------------------------------------------------------

def test_group_against_dict_brute_force():
    rng = np.random.default_rng(8)
    for (T, k, E) in [(1, 2, 8), (8, 16, 896), (37, 4, 11)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        offs, tok, slot, n = orc.group(ids, E)
        lists = {}
        for t in range(T):
            for j in range(k):
                lists.setdefault(int(ids[t, j]), []).append((t, j))
        assert n == len(lists)
        for e in range(E):
            seg = list(zip(tok[offs[e]:offs[e + 1]], slot[offs[e]:offs[e + 1]]))
            assert seg == lists.get(e, [])


# ---- RMSNorm -------------------------------------------------------------------

def test_rmsnorm_bf16_closed_form():
    import torch
    x = synth.normal_bf16(synth.key(1, 4, 0, 5, 0), 3 * 512, 3.0).reshape(3, 512)
    got = orc.rmsnorm_bf16(x, 1e-6)
    xf = bf16_bits_to_f64(x)
    ref = xf / np.sqrt((xf ** 2).mean(axis=1, keepdims=True) + 1e-6)
    ref_bits = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref_bits)
    # a constant row normalises to +-1 (up to eps)
    c = np.full((1, 64), 0x4040, dtype=np.uint16)  # 3.0
    assert np.all(orc.rmsnorm_bf16(c, 0.0) == 0x3F80)


# ---- whole layer: brute force on the tiny workload ------------------------------

def tiny_layer(seed=0, k=2, zero_codes=False, n_shared=1):
    H, I, E, Is = 256, 64, 8, 64
    spans = synth.expert_spans(seed, 0, 0, 0, E, H, I)
    if zero_codes:
        for e in range(E):
            for t, a in enumerate(split_span(spans[e], H, I)):
                if t % 2 == 0:
                    a[...] = 0
    router = synth.router(seed, 0, 0, E, H)
    shared = [synth.shared(seed, 0, 0, s, H, Is) for s in range(n_shared)]
    L = orc.Layer(H, E, k, I, Is, router, shared, lambda l, e: spans[e])
    return L, spans, router, shared


def brute_force_layer(spans, router, shared, x_bits, k, residual=None, I=64):
    H = x_bits.shape[-1]
    out = []
    for t in range(x_bits.shape[0]):
        x = bf16_bits_to_f64(x_bits[t])
        logits = router.astype(np.float64) @ x
        E = logits.size
        ys = [ffn_numpy(spans[e], H, I, x) for e in range(E)]
        best = sorted(range(E), key=lambda e: (-logits[e], e))[:k]
        w = np.exp(logits[best] - logits[best].max()); w /= w.sum()
        y = sum(wi * ys[e] for wi, e in zip(w, best))
        y = y + sum(shared_numpy(*s, x) for s in shared)
        if residual is not None:
            y = y + bf16_bits_to_f64(residual[t])
        out.append((y, best, w))
    return out


def test_tiny_layer_brute_force_all_experts():
    L, spans, router, shared = tiny_layer()
    x = np.stack([synth.token(0, 0, t, 256) for t in range(4)])
    res = np.stack([synth.token(0, 0, t, 256, kind=synth.gen.KIND_RESIDUAL) for t in range(4)])
    r = orc.moe_layer(L, x, residual=res)
    ref = brute_force_layer(spans, router, shared, x, 2, residual=res)
    for t in range(4):
        y, best, w = ref[t]
        assert list(r["ids"][t]) == best
        assert np.allclose(r["w"][t], w, rtol=1e-12)
        assert np.allclose(r["out"][t], y, rtol=1e-10, atol=1e-9 * np.abs(y).max())
        assert np.allclose(r["routed"][t] + r["shared"][t] + bf16_bits_to_f64(res[t]),
                           r["out"][t], rtol=1e-14, atol=1e-12)


def test_all_zero_codes_leave_shared_only():
    L, spans, router, shared = tiny_layer(zero_codes=True)
    x = synth.token(0, 0, 0, 256)[None, :]
    r = orc.moe_layer(L, x)
    assert np.all(r["routed"] == 0.0)
    ref = shared_numpy(*shared[0], bf16_bits_to_f64(x[0]))
    assert np.allclose(r["out"][0], ref, rtol=1e-12, atol=1e-12)


def test_k_equals_e_is_dense_softmax_moe():
    L, spans, router, shared = tiny_layer(k=8)
    x = synth.token(0, 0, 5, 256)[None, :]
    r = orc.moe_layer(L, x)
    xd = bf16_bits_to_f64(x[0])
    logits = router.astype(np.float64) @ xd
    p = np.exp(logits - logits.max()); p /= p.sum()
    dense = sum(p[e] * ffn_numpy(spans[e], 256, 64, xd) for e in range(8))
    assert np.allclose(r["routed"][0], dense, rtol=1e-10, atol=1e-9 * np.abs(dense).max())


def test_two_shared_experts_add_unweighted():
    L, spans, router, shared = tiny_layer(n_shared=2)
    x = synth.token(0, 0, 2, 256)[None, :]
    r = orc.moe_layer(L, x)
    xd = bf16_bits_to_f64(x[0])
    ref = shared_numpy(*shared[0], xd) + shared_numpy(*shared[1], xd)
    assert np.allclose(r["shared"][0], ref, rtol=1e-12, atol=1e-12)


def test_stack_composes_norm_layer_and_residual():
    import torch
    H = 256
    layers, parts = [], []
    for l in range(2):
        spans = synth.expert_spans(0, 0, l, 0, 8, H, 64)
        router = synth.router(0, 0, l, 8, H)
        shared = [synth.shared(0, 0, l, 0, H, 64)]
        layers.append(orc.Layer(H, 8, 2, 64, 64, router, shared,
                                (lambda sp: (lambda ly, e: sp[e]))(spans), layer=l))
        parts.append((spans, router, shared))
    x = np.stack([synth.token(0, 0, t, H) for t in range(2)])
    r = orc.moe_stack(layers, x, 1e-6)
    cur = x.copy()
    for l, (spans, router, shared) in enumerate(parts):
        xf = bf16_bits_to_f64(cur)
        xn = xf / np.sqrt((xf ** 2).mean(axis=1, keepdims=True) + 1e-6)
        xn_bits = torch.from_numpy(xn).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        ref = brute_force_layer(spans, router, shared, xn_bits, 2, residual=cur)
        nxt = np.stack([ref[t][0] for t in range(2)])
        for t in range(2):
            assert list(r["ids"][l, t]) == ref[t][1]
        if l == len(parts) - 1:
            assert np.allclose(r["last"], nxt, rtol=1e-10, atol=1e-9 * np.abs(nxt).max())
        cur = torch.from_numpy(nxt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r["x"], cur)
