// The fused elementwise epilogue: one scalar function of the f32 accumulator
// (and, for the bias ops, of the column's bias), applied per output element
// before the conversion to D's type.  It follows "Explicit CUDA tile
// patterns", section "Scalar compositions" (TVM TIRx): a caller-chosen scalar
// function such as silu_affine(x, scale, bias) = x / (1 + exp(-x)) * scale +
// bias, inlined at each register element.  AFFINE (x * alpha + beta) carries
// a per-tensor scale, e.g. the global scale of NVFP4 operands.
#pragma once

#include <cstdint>

namespace tg {

// Epilogue parameters as the kernels see them (op codes are TG_EPI_*).
struct Epi {
  int op;
  float alpha;
  float beta;
  const float* bias;   // device f32 [N] for the column-bias ops
};

enum : int {
  kEpiNone = 0,
  kEpiAddScalar = 1,
  kEpiSiluAffine = 2,
  kEpiBiasCol = 3,
  kEpiBiasColSilu = 4,
  kEpiAffine = 5,
};

__host__ __device__ constexpr bool epi_uses_bias(int op) {
  return op == kEpiBiasCol || op == kEpiBiasColSilu;
}

#ifdef __CUDACC__
// silu(x) = x / (1 + e^(-x)) with CUDA's fast exponential and divide: a few
// ulp of relative error (both intrinsics are documented to within 2 ulp plus,
// for __expf, ~1.16|x| ulp), which is far inside the product's own error
// bound.  Large negative x give e^(-x) = inf and a result of -0.
__device__ __forceinline__ float silu_f32(float x) {
  return __fdividef(x, 1.0f + __expf(-x));
}

// The ops other than NONE / ADD_SCALAR, on one value; `b` is the column's
// bias (unused by SILU_AFFINE and AFFINE).  NONE and ADD_SCALAR are applied by the
// stores themselves, as acc + (0 or alpha).
__device__ __forceinline__ float apply_epi_general(int op, float alpha, float beta, float x,
                                                   float b) {
  if (op == kEpiSiluAffine) return silu_f32(x) * alpha + beta;
  if (op == kEpiAffine) return x * alpha + beta;
  if (op == kEpiBiasCol) return x + b;
  return silu_f32(x + b);
}
#endif

}  // namespace tg
