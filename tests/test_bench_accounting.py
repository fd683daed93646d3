"""The roofline numerators: the bench's algorithmic byte counts against the
closed forms of the K3 layer. MXFP4 costs 17/32 B a weight (4 bits plus one
8-bit scale per 32 weights; kimi-k3-in-c blog, section 先把账算明白), so a
SwiGLU expert of 3 x 7168 x 1536 weights is 17,547,264 B, two thirds of it
gate and up. The router is fp32 [896][7168];
the two shared experts are bf16 SwiGLU FFNs of intermediate 1536.
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402

K3 = synth.WORKLOADS[1]
H, I, E, k = 7168, 1536, 896, 16


def test_k3_workload_shape():
    assert (K3.H, K3.I, K3.E, K3.k, K3.n_shared, K3.Is, K3.T) == (H, I, E, k, 2, 1536, 1)


def test_expert_bytes():
    weights = 3 * H * I
    assert synth.span_bytes(H, I) == weights * 17 // 32 == 17_547_264
    assert 2 * I * H * 17 // 32 == 11_698_176  # gate + up: two thirds of the span


def test_batch1_layer_bytes():
    router = E * H * 4
    shared = 2 * 3 * 1536 * H * 2
    assert (router, shared) == (25_690_112, 132_120_576)
    weights = router + shared + k * 17_547_264
    assert weights == 438_566_912
    # plus x in and out, bf16
    assert bench.layer_bytes(K3, 16, 1) == weights + 2 * H * 2


def test_batch1_gateup_launch_bytes():
    routed = 16 * 11_698_176 + H * 2 + k * I * 4          # experts, x in, h out
    shared = 2 * 2 * 1536 * H * 2 + 2 * 1536 * 4           # gate/up rows, their h
    assert bench.gateup_bytes(K3, 16, 1) == routed
    assert bench.gateup_bytes(K3, 16, 1, with_shared=True) == routed + shared == 275_376_128


def test_bytes_grow_with_distinct_experts_only():
    # a second token that reuses every expert adds only its activations
    one = bench.layer_bytes(K3, 16, 1)
    assert bench.layer_bytes(K3, 16, 2) - one == 2 * H * 2
    assert bench.layer_bytes(K3, 17, 1) - one == 17_547_264


def test_batch1_planes_phase_gateup_bytes():
    # the one-token gate/up phase of an exact-planes handle: the routed experts,
    # x's 4 E4M3 planes with one scale byte per 32, the gate and up sums of 8
    # parts of K (fp32); beside them the shared gate/up rows, x (bf16), their h
    routed = 16 * 11_698_176 + 4 * (H + H // 32) + 8 * k * 2 * I * 4
    shared = 2 * 2 * 1536 * H * 2 + H * 2 + 2 * 1536 * 4
    assert bench.mx8_phase_gateup_bytes(K3, 16) == routed + shared == 276_880_256
