"""Host checks of the tcgen05 operand encodings (csrc/umma.cuh), compiled
with g++ from the same header the kernels use.

The fields are checked against the bit positions of the PTX ISA's tables for
tcgen05 (the shared memory matrix descriptor and the instruction descriptor
of .kind::f16), and the K-major tile layout against the canonical
no-swizzle form: 8 x 16-byte core matrices stored as 128 contiguous bytes,
neighbours along K `LBO` bytes apart and along the rows `SBO` bytes apart.
It also checks the property the kernel relies on for safety: whichever way
the two offsets are read, one MMA's operand stays inside its 16-column
block of the stage.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "mxfp4_routed_expert_top_gb300", "csrc")

DRIVER = r"""
#define __host__
#define __device__
#include <cstdio>
#include "umma.cuh"
int main() {
  using namespace dfm::umma;
  printf("LBO %u SBO %u\n", kLBO, kSBO);
  const unsigned addrs[3] = {0x400u, 0x11A30u, 0x3FFF0u};
  for (unsigned a : addrs) printf("D %u %llu\n", a, (unsigned long long)smem_desc(a, kLBO, kSBO));
  for (unsigned a : addrs) printf("S %u %llu\n", a, (unsigned long long)smem_desc_sw128(a));
  const int ns[5] = {16, 32, 48, 64, 256};
  for (int n : ns) printf("I %d %d %u\n", 128, n, idesc_bf16_f32(128, n));
  for (int n : ns) printf("F %d %d %u\n", 128, n, idesc_f16_f32(128, n));
  for (int n : ns)
    for (int a = 0; a < 4; ++a)
      for (int b = 0; b < 4; ++b)
        printf("X %d %d %d %d %u\n", 128, n, a, b, idesc_mxf8f6f4_e2m1_e4m3(128, n, a, b));
  const int rows[4] = {16, 32, 64, 128};
  for (int R : rows)
    for (int r = 0; r < R; ++r)
      for (int k = 0; k < 64; ++k) printf("K %d %d %d %u\n", R, r, k, kmajor_offset(R, r, k));
  return 0;
}
"""


@pytest.fixture(scope="module")
def enc(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no g++")
    d = tmp_path_factory.mktemp("umma")
    src, exe = d / "drv.cpp", d / "drv"
    src.write_text(DRIVER)
    subprocess.run([gxx, "-std=c++17", "-O0", "-I" + CSRC, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    res = {"D": {}, "S": {}, "I": {}, "F": {}, "K": {}, "X": {}}
    for line in out.splitlines():
        f = line.split()
        if f[0] == "LBO":
            res["LBO"], res["SBO"] = int(f[1]), int(f[3])
        elif f[0] in ("D", "S"):
            res[f[0]][int(f[1])] = int(f[2])
        elif f[0] in ("I", "F"):
            res[f[0]][(int(f[1]), int(f[2]))] = int(f[3])
        elif f[0] == "X":
            res["X"][tuple(int(v) for v in f[1:5])] = int(f[5])
        else:
            res["K"].setdefault(int(f[1]), {})[(int(f[2]), int(f[3]))] = int(f[4])
    return res


def bits(v, lo, hi):
    return (v >> lo) & ((1 << (hi - lo)) - 1)


def test_smem_descriptor_fields(enc):
    for a, d in enc["D"].items():
        assert bits(d, 0, 14) == (a >> 4) & 0x3FFF          # start address >> 4
        assert bits(d, 16, 30) == enc["LBO"] >> 4            # leading byte offset >> 4
        assert bits(d, 32, 46) == enc["SBO"] >> 4            # stride byte offset >> 4
        assert bits(d, 46, 48) == 1                          # descriptor version (sm_100)
        assert bits(d, 49, 52) == 0                          # base offset
        assert bits(d, 52, 53) == 0                          # relative offset mode
        assert bits(d, 61, 64) == 0                          # no swizzle
        assert bits(d, 14, 16) == 0 and bits(d, 30, 32) == 0 and bits(d, 53, 61) == 0


def test_swizzled_descriptor_fields(enc):
    for a, d in enc["S"].items():
        assert bits(d, 0, 14) == (a >> 4) & 0x3FFF
        assert bits(d, 16, 30) == 1                          # leading offset unused: 1
        assert bits(d, 32, 46) == 1024 >> 4                  # 8-row atom of 128-byte rows
        assert bits(d, 46, 48) == 1
        assert bits(d, 49, 53) == 0                          # base offset 0: 1024-aligned stages
        assert bits(d, 61, 64) == 2                          # 128-byte swizzle


def test_instruction_descriptor_fields(enc):
    for (M, N), v in enc["I"].items():
        assert bits(v, 0, 4) == 0        # dense, no saturation
        assert bits(v, 4, 6) == 1        # D: f32
        assert bits(v, 7, 10) == 1       # A: bf16
        assert bits(v, 10, 13) == 1      # B: bf16 (same type as A)
        assert bits(v, 13, 15) == 0      # no negation
        assert bits(v, 15, 17) == 0      # A and B K-major
        assert bits(v, 17, 23) == N >> 3
        assert bits(v, 23, 24) == 0
        assert bits(v, 24, 29) == M >> 4
        assert bits(v, 29, 32) == 0
        assert M == 128 and N % 16 == 0 and 16 <= N <= 256   # valid cta_group::1 shapes


def test_instruction_descriptor_f16(enc):
    for (M, N), v in enc["F"].items():
        assert bits(v, 4, 6) == 1        # D: f32
        assert bits(v, 7, 13) == 0       # A and B: f16 (the same type)
        assert bits(v, 17, 23) == N >> 3 and bits(v, 24, 29) == M >> 4
        assert v & ~((0x3 << 4) | (0x3F << 17) | (0x1F << 24)) == 0


def test_instruction_descriptor_block_scaled(enc):
    """kind::mxf8f6f4.block_scale with E2M1 A (the weights) and E4M3 B (the
    activations): the block-scaled descriptor moves M to bits 27-28 (M >> 7)
    and puts the two scale-factor ids (which byte of each 32-bit scale word
    in tensor memory the MMA takes) at bits 4-5 (B) and 29-30 (A)."""
    assert len(enc["X"]) == 5 * 16
    for (M, N, a, b), v in enc["X"].items():
        assert bits(v, 0, 4) == 0        # dense
        assert bits(v, 4, 6) == b        # B scale factor id
        assert bits(v, 6, 7) == 0
        assert bits(v, 7, 10) == 5       # A: E2M1
        assert bits(v, 10, 13) == 0      # B: E4M3
        assert bits(v, 13, 15) == 0      # no negation
        assert bits(v, 15, 17) == 0      # A and B K-major (the only form for E2M1)
        assert bits(v, 17, 23) == N >> 3
        assert bits(v, 23, 24) == 1      # scale type E8M0
        assert bits(v, 24, 27) == 0
        assert bits(v, 27, 29) == M >> 7
        assert bits(v, 29, 31) == a      # A scale factor id
        assert bits(v, 31, 32) == 0      # K = 32 a step (dense)


def test_kmajor_layout(enc):
    L, S = enc["LBO"], enc["SBO"]
    for R, off in enc["K"].items():
        vals = np.array(sorted(off.values()))
        # a bijection onto [0, 2 R 64) in steps of one element
        assert np.array_equal(vals, np.arange(0, R * 128, 2))
        for (r, k), o in off.items():
            blk = (k // 16) * R * 32
            # core matrix: 8 rows x 8 elements, 128 contiguous bytes, row-major
            assert (o - blk) % 128 == (r % 8) * 16 + (k % 8) * 2
            if k % 16 < 8:
                assert off[(r, k + 8)] - o == L      # neighbour along K
            if r + 8 < R:
                assert off[(r + 8, k)] - o == S      # neighbour along the rows
            # every element of one MMA (16 K-columns) lies in its block
            assert blk <= o < blk + R * 32


def test_operand_reads_stay_in_block_either_way(enc):
    # the furthest byte one MMA can read from a block start, with the offsets
    # as intended and swapped, stays inside the R x 16 block (R * 32 bytes)
    L, S = enc["LBO"], enc["SBO"]
    for R in enc["K"]:
        for lead, stride in ((L, S), (S, L)):
            far = (R // 8 - 1) * stride + 1 * lead + 127
            assert far < R * 32, (R, lead, stride)
