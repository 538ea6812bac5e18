// Operand kinds of the GEMM kernels and their K geometry, shared by host and
// device code.
//
// kKindBf16: dense bf16 (.kind::f16).  Block-scaled kinds ("tcgen05.mma",
// TVM TIRx tile-operation guide, section "Weight-stationary and block
// scaling": .block_scale with .scale_vec::1X / 2X / 4X):
//   kKindMxf8  E4M3 operands, one E8M0 scale per 32 K   (.kind::mxf8f6f4, 1X)
//   kKindMxf4  packed E2M1, one E8M0 scale per 32 K     (.kind::mxf4nvf4, 2X)
//   kKindNvf4  packed E2M1, one UE4M3 scale per 16 K    (.kind::mxf4nvf4, 4X)
#pragma once

namespace tg {

enum : int { kKindBf16 = 0, kKindMxf8 = 1, kKindMxf4 = 2, kKindNvf4 = 3 };

// Scales per row that one MMA reads (the .scale_vec width); 0 for bf16.
__host__ __device__ constexpr int scale_vec_of(int kind) {
  return kind == kKindMxf8 ? 1 : kind == kKindMxf4 ? 2 : kind == kKindNvf4 ? 4 : 0;
}

// K elements that share one scale byte.
__host__ __device__ constexpr int scale_block_of(int kind) { return kind == kKindNvf4 ? 16 : 32; }

// K elements in one 128-byte stage row (one element per byte for E4M3, two
// for packed E2M1).
__host__ __device__ constexpr int stage_k_of(int kind) {
  return kind == kKindBf16 ? 64 : kind == kKindMxf8 ? 128 : 256;
}

}  // namespace tg
