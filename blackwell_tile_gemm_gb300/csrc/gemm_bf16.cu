// Dense bf16 GEMM configurations (kind::f16, f32 accumulation).
//
//   single CTA : 128 x 256 tiles, 4-stage ring of 48 KB, two 256-column
//                accumulators in tensor memory (all 512 columns).
//   CTA pair   : 256 x 256 tiles per cluster of two (cta_group::2), each CTA
//                stages 128 rows of A and 128 rows of B per stage (32 KB),
//                6-stage ring, two accumulators per CTA.
//   multicast  : clusters of two CTA pairs on vertically adjacent tiles; each
//                CTA loads a 64-row quarter of the shared B tile and
//                multicasts it to its counterpart in the other pair.
#include "gemm_launch.cuh"

namespace tg {

namespace {
// m-tiles per band of the persistent tile order.
constexpr int kRasterGroup = 8;
using CfgF32 = GemmCfg<1, kKindBf16, 256, 2, 4, false>;
using CfgBf16 = GemmCfg<1, kKindBf16, 256, 2, 4, true>;
using CfgPairF32 = GemmCfg<2, kKindBf16, 256, 2, 6, false>;
using CfgPairBf16 = GemmCfg<2, kKindBf16, 256, 2, 6, true>;
// Clusters of two CTA pairs multicasting the shared B tile (TG_FLAG_MULTICAST).
using CfgPairMcF32 = GemmCfg<2, kKindBf16, 256, 2, 6, false, true>;
using CfgPairMcBf16 = GemmCfg<2, kKindBf16, 256, 2, 6, true, true>;
}  // namespace

int launch_gemm_bf16_impl(const void* A, int64_t lda, const void* B, int64_t ldb, void* D,
                          int64_t ldd, int M, int N, int K, int d_dtype, const Epi& epi,
                          bool pair, bool mcast, cudaStream_t stream, DeviceCtx* ctx) {
  constexpr int BN = 256;
  const int g = pair ? 2 : 1;
  const int b_rows = BN / g;
  CUtensorMap tA, tB;
  int rc = make_tensor_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, 64, 128,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  const int b_box = pair && mcast ? b_rows / 2 : b_rows;
  rc = make_tensor_map_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, ldb * 2, 64, b_box,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.num_m_tiles = ceil_div_i(M, 128 * g);
  a.num_n_tiles = ceil_div_i(N, BN);
  a.num_k_blocks = ceil_div_i(K, 64);
  a.D = D;
  a.ldd = ldd;
  a.epi = epi;
  a.raster_group = kRasterGroup;
  a.status = ctx->status;
  a.timeout_ns = wait_timeout_ns();
  const bool bf16_out = d_dtype == TG_D_BF16;
  if (!pair)
    return bf16_out ? launch_gemm_cfg<CfgBf16>(tA, tB, tA, tB, a, stream, ctx)
                    : launch_gemm_cfg<CfgF32>(tA, tB, tA, tB, a, stream, ctx);
  if (mcast)
    return bf16_out ? launch_gemm_cfg<CfgPairMcBf16>(tA, tB, tA, tB, a, stream, ctx)
                    : launch_gemm_cfg<CfgPairMcF32>(tA, tB, tA, tB, a, stream, ctx);
  return bf16_out ? launch_gemm_cfg<CfgPairBf16>(tA, tB, tA, tB, a, stream, ctx)
                  : launch_gemm_cfg<CfgPairF32>(tA, tB, tA, tB, a, stream, ctx);
}

int bf16_tail_split(int64_t M, int64_t N, int64_t K, bool pair, DeviceCtx* ctx) {
  const int g = pair ? 2 : 1;
  const int num_tiles = ceil_div_i(M, 128 * g) * ceil_div_i(N, 256);
  const int units_max =
      pair ? gemm_units_for_device<CfgPairF32>(ctx) : gemm_units_for_device<CfgF32>(ctx);
  if (units_max < 0) return -TG_ERR_CUDA;
  int W = 0, R = 0;
  return pair ? tail_split_for<CfgPairF32>(num_tiles, ceil_div_i(K, 64), units_max, &W, &R)
              : tail_split_for<CfgF32>(num_tiles, ceil_div_i(K, 64), units_max, &W, &R);
}

// ---------------------------------------------------------------------------
// K == 0: D = epilogue(0)
// ---------------------------------------------------------------------------

namespace {
__global__ void fill_kernel(void* D, int64_t ldd, int64_t M, int64_t N, int bf16_out, Epi epi) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i % N;
    float y = 0.0f;
    if (epi.op == kEpiAddScalar)
      y = epi.alpha;
    else if (epi.op != kEpiNone)
      y = apply_epi_general(epi.op, epi.alpha, epi.beta, 0.0f,
                            epi_uses_bias(epi.op) ? epi.bias[c] : 0.0f);
    if (bf16_out)
      reinterpret_cast<uint16_t*>(D)[r * ldd + c] =
          static_cast<uint16_t>(pack_bf16x2(y, y) & 0xFFFFu);
    else
      reinterpret_cast<float*>(D)[r * ldd + c] = y;
  }
}
}  // namespace

int launch_fill_epilogue(void* D, int64_t ldd, int64_t M, int64_t N, int d_dtype, const Epi& epi,
                         cudaStream_t stream) {
  const int64_t total = M * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(D, ldd, M, N,
                                                                 d_dtype == TG_D_BF16, epi);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

}  // namespace tg
