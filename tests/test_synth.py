"""The seeded input generator: definition, determinism, distributions."""
import numpy as np

import synth


def test_splitmix64_published_sequence():
    # SplitMix64 seeded with 0 (Vigna's splitmix64.c) starts with these words
    expect = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [synth.at(0, i) for i in range(3)] == expect
    assert list(synth.words(0, 0, 3)) == expect


def test_random_access_and_determinism():
    k = synth.key(7, 1, 2, synth.gen.KIND_ROUTER, 0)
    a = synth.normal_f32(k, 1000, 1.0)
    b = synth.normal_f32(k, 400, 1.0, first=600)
    assert np.array_equal(a[600:], b)
    assert np.array_equal(a, synth.normal_f32(k, 1000, 1.0))
    assert synth.key(7, 1, 2, 1, 0) != synth.key(7, 1, 2, 1, 1)
    assert synth.key(7, 1, 2, 1, 0) != synth.key(8, 1, 2, 1, 0)


def test_normal_moments():
    z = synth.normal_f64(synth.key(0, 9, 0, 5, 0), 400000, 1.0)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    assert abs((z ** 4).mean() - 3.0) < 0.05
    # tail mass beyond 3 sigma ~ 0.27%
    assert 0.0020 < np.mean(np.abs(z) > 3) < 0.0034


def test_bf16_is_rne_of_fp32():
    import torch
    k = synth.key(0, 9, 0, 5, 1)
    f = synth.normal_f32(k, 5000, 1.0)
    b = synth.normal_bf16(k, 5000, 1.0)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)


def test_expert_span_distributions():
    H, I = 1024, 512
    sp = synth.expert_spans(3, 1, 0, 10, 2, H, I)
    assert sp.shape == (2, 3 * (H * I // 2 + H * I // 32))
    q = sp[0, :H * I // 2]
    codes = np.concatenate([q & 15, q >> 4])
    counts = np.bincount(codes, minlength=16)
    exp = codes.size / 16
    assert ((counts - exp) ** 2 / exp).sum() < 60  # chi-square, 15 dof
    s = sp[0, H * I // 2:H * I // 2 + H * I // 32]
    assert s.min() >= 119 and s.max() <= 127
    assert set(np.unique(s)) == set(range(119, 128))
    # experts differ; the same expert regenerates identically
    assert not np.array_equal(sp[0], sp[1])
    assert np.array_equal(sp[1], synth.expert_spans(3, 1, 0, 11, 1, H, I)[0])


def test_token_redraws_are_independent():
    a = synth.token(0, 1, 5, 256, redraw=0)
    b = synth.token(0, 1, 5, 256, redraw=1)
    assert not np.array_equal(a, b)


def test_f64_to_bf16_bits_matches_torch():
    import torch
    a = np.concatenate([synth.normal_f64(synth.key(1, 2, 0, 5, 3), 4000, 3.0),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, -2.5e-3]])
    ref = (torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
           .view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(synth.f64_to_bf16_bits(a), ref)


def test_token_stream_window_moments_and_correlation():
    H, rho = 7168, 0.7
    full = synth.token_stream(4, 3, 0, 12, H, rho)
    assert np.array_equal(synth.token_stream(4, 3, 5, 4, H, rho), full[5:9])
    x = (full.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    # every token N(0, 1); neighbours correlated rho, two apart rho^2
    assert np.all(np.abs(x.var(axis=1) - 1.0) < 0.06)
    c1 = np.mean([np.corrcoef(x[i], x[i + 1])[0, 1] for i in range(11)])
    c2 = np.mean([np.corrcoef(x[i], x[i + 2])[0, 1] for i in range(10)])
    assert abs(c1 - rho) < 0.02 and abs(c2 - rho * rho) < 0.02
    ind = synth.token_stream(4, 3, 0, 6, H, 0.0)
    y = (ind.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(np.corrcoef(y[0], y[1])[0, 1]) < 0.05
