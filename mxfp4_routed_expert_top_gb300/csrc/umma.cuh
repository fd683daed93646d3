// umma.cuh — encodings for the 5th-generation tensor core MMA (tcgen05.mma)
// of sm_100-family GPUs: shared-memory matrix descriptors and the
// instruction descriptors of kind::f16 and kind::mxf8f6f4.block_scale. Host
// and device, so that the host tests can check them field by field.
//
// Operands here are K-major and unswizzled ("interleaved"): a matrix of R
// rows x 16 K-columns of 16-bit elements is made of core matrices of
// 8 rows x 16 bytes (8 elements), each stored as 128 contiguous bytes. The
// descriptor gives the byte distance between core matrices that are
// neighbours along K (leading dimension offset) and along the rows (stride
// dimension offset).
#pragma once

#include <stdint.h>

namespace dfm {
namespace umma {

// Shared-memory matrix descriptor (64 bits):
//   [0,14)  start address >> 4      [16,30) leading dimension offset >> 4
//   [32,46) stride dimension offset >> 4   [46,48) version = 1
//   [49,52) base offset = 0   [52] offset mode = 0   [61,64) layout = 0 (no swizzle)
__host__ __device__ inline uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// The same for a K-major operand in the 128-byte swizzle layout (rows of 128
// bytes, 8-row atoms of 1024 bytes, 16-byte chunks XOR-permuted by the row
// within the atom): the stride dimension offset is the atom (1024 bytes), the
// leading dimension offset is unused (1 by convention), layout type 2. The
// start address of K step j (16 elements of 16 bits) is the base + 32 j.
__host__ __device__ inline uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 (32 bits), dense, fp32 D,
// bf16 A and B, both K-major:
//   [4,6) D format (1 = f32)  [7,10) A format (1 = bf16)  [10,13) B format
//   [15] A major (0 = K)  [16] B major  [17,23) N >> 3  [24,29) M >> 4
__host__ __device__ inline uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// The same with f16 A and B (A and B formats 0).
__host__ __device__ inline uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of tcgen05.mma kind::mxf8f6f4.block_scale (32
// bits), dense, fp32 D, E2M1 A (the weights) and E4M3 B (the activations),
// both K-major, E8M0 scale factors:
//   [4,6) B scale factor id (the byte of the 32-bit scale word in tensor
//   memory)  [7,10) A format (5 = E2M1)  [10,13) B format (0 = E4M3)
//   [15] A major  [16] B major  [17,23) N >> 3  [23] scale type (1 = E8M0)
//   [27,29) M >> 7  [29,31) A scale factor id
__host__ __device__ inline uint32_t idesc_mxf8f6f4_e2m1_e4m3(int M, int N, int a_sf, int b_sf) {
  return ((uint32_t)(b_sf & 3) << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
         (1u << 23) | ((uint32_t)(M >> 7) << 27) | ((uint32_t)(a_sf & 3) << 29);
}

// Byte offset of element (r, k) (16-bit elements) in a K-major tile of `rows`
// rows x 64 K-columns laid out as 4 blocks of 16 K-columns, each block
// [rows/8 core-matrix rows][2 core matrices along K][8 rows][16 bytes]:
// block stride rows*32 bytes, leading dimension offset 128, stride dimension
// offset 256.
__host__ __device__ inline uint32_t kmajor_offset(int rows, int r, int k) {
  return (uint32_t)((k >> 4) * rows * 32 + (r >> 3) * 256 + ((k >> 3) & 1) * 128 + (r & 7) * 16 +
                    (k & 7) * 2);
}
constexpr uint32_t kLBO = 128, kSBO = 256;

}  // namespace umma
}  // namespace dfm
