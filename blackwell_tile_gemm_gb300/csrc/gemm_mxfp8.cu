// Block-scaled MXFP8 GEMM (kind::mxf8f6f4 .block_scale .scale_vec::1X):
// E4M3 operands, one E8M0 scale per 32 K elements per row, f32 accumulation.
//
// Scale factors reach tensor memory as "tcgen05.mma" (section
// "Weight-stationary and block scaling") lays them out: scale row r sits in
// TMEM lane r % 32, byte column 4 * (r / 32) + sf, replicated in the four
// 32-lane slabs; the scale-factor id in the instruction descriptor selects the
// byte.  tcgen05.cp .32x128b.warpx4 ("Explicit CUDA tile patterns", section
// "TMEM transfers": warpx4 adds four replicas 32 lanes apart) copies 32 rows
// of 16 bytes, so the shared-memory image of 128 scale rows x 4 K-blocks is
// 512 bytes with byte (16 * l + 4 * j + k) = scale of row 32 * j + l, block k.
//
// sf_repack_kernel writes those 512-byte images from the caller's natural
// [rows, K/32] byte arrays into the workspace, ordered [K group][128-row
// block]; the GEMM then fetches one image per operand and stage with TMA.
//
// Configurations: single CTA 128 x 256 tiles, 4 stages of 49.5 KB, one
// 256-column accumulator plus 12 scale columns per stage; CTA pair 256 x 256
// tiles, 6 stages of 33.5 KB per CTA.
#include "gemm_launch.cuh"

namespace tg {

namespace {
// m-tiles per band of the persistent tile order.
constexpr int kRasterGroup = 8;

using CfgMxF32 = GemmCfg<1, true, 256, 1, 4, false>;
using CfgMxBf16 = GemmCfg<1, true, 256, 1, 4, true>;
using CfgMxPairF32 = GemmCfg<2, true, 256, 1, 6, false>;
using CfgMxPairBf16 = GemmCfg<2, true, 256, 1, 6, true>;
using CfgMxPairMcF32 = GemmCfg<2, true, 256, 1, 6, false, true>;
using CfgMxPairMcBf16 = GemmCfg<2, true, 256, 1, 6, true, true>;

struct SfImage {
  const uint8_t* src;   // [rows, kblocks] bytes, row stride ld
  int64_t ld;
  int rows;
  int blocks;           // 128-row blocks per K group in the image
  uint32_t* dst;        // [num_kg][blocks][128] words
};

// Image word (4*l + j) of 128-row block b, K group g holds the scales of row
// 128*b + 32*j + l for K blocks 4*g .. 4*g+3 (low byte first); rows or K
// blocks past the end are zero.  Work unit: one warp per (image, block,
// quad of K groups, l-octet).  Lane (4*l' + j) reads the 16 scale bytes of
// K groups 4*quad .. 4*quad+3 of its row and writes one word into each of
// those four images, so that each warp store covers 32 consecutive words
// (128 bytes) of one image.
__global__ void sf_repack_kernel(SfImage a, SfImage b, int kblocks, int num_kg) {
  const int quads = (num_kg + 3) / 4;
  const int64_t warps_a = static_cast<int64_t>(a.blocks) * quads * 4;
  const int64_t warps_b = static_cast<int64_t>(b.blocks) * quads * 4;
  const int lane = threadIdx.x & 31;
  const int64_t warps_per_grid = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t wid = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
       wid < warps_a + warps_b; wid += warps_per_grid) {
    const bool is_a = wid < warps_a;
    const SfImage& s = is_a ? a : b;
    const int64_t w = is_a ? wid : wid - warps_a;
    const int octet = static_cast<int>(w & 3);
    const int64_t bq = w >> 2;
    const int quad = static_cast<int>(bq % quads);
    const int blk = static_cast<int>(bq / quads);
    const int l = 8 * octet + (lane >> 2), j = lane & 3;
    const int row = blk * 128 + 32 * j + l;
    uint32_t v[4] = {0, 0, 0, 0};
    if (row < s.rows) {
      const uint8_t* src = s.src + static_cast<int64_t>(row) * s.ld;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int kb = 16 * quad + t;
        if (kb < kblocks) v[t >> 2] |= static_cast<uint32_t>(__ldg(src + kb)) << (8 * (t & 3));
      }
    }
    const int64_t per_kg = static_cast<int64_t>(s.blocks) * 128;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kg = 4 * quad + t;
      if (kg < num_kg) s.dst[kg * per_kg + blk * 128 + 4 * l + j] = v[t];
    }
  }
}

struct MxPlan {
  int num_m_tiles, num_n_tiles, num_kg, sfa_blocks, sfb_blocks;
};

MxPlan plan_mx(int64_t M, int64_t N, int64_t K, bool pair) {
  const int g = pair ? 2 : 1;
  MxPlan p{};
  p.num_m_tiles = ceil_div_i(M, 128 * g);
  p.num_n_tiles = ceil_div_i(N, 256);
  p.num_kg = ceil_div_i(K, 128);
  p.sfa_blocks = p.num_m_tiles * g;
  p.sfb_blocks = p.num_n_tiles * 2;
  return p;
}

}  // namespace

size_t mxfp8_workspace_bytes(int64_t M, int64_t N, int64_t K, bool pair) {
  const MxPlan p = plan_mx(M, N, K, pair);
  return static_cast<size_t>(p.sfa_blocks + p.sfb_blocks) * p.num_kg * 512u;
}

int launch_gemm_mxfp8_impl(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int M, int N, int K, int d_dtype,
                           const Epi& epi, bool pair, bool mcast, uint8_t* sf_workspace,
                           cudaStream_t stream, DeviceCtx* ctx) {
  const MxPlan pl = plan_mx(M, N, K, pair);
  const int g = pair ? 2 : 1;
  uint8_t* img_a = sf_workspace;
  uint8_t* img_b = sf_workspace + static_cast<size_t>(pl.sfa_blocks) * pl.num_kg * 512u;

  SfImage sa{static_cast<const uint8_t*>(SFA), ld_sfa, M, pl.sfa_blocks,
             reinterpret_cast<uint32_t*>(img_a)};
  SfImage sb{static_cast<const uint8_t*>(SFB), ld_sfb, N, pl.sfb_blocks,
             reinterpret_cast<uint32_t*>(img_b)};
  const int64_t warps =
      static_cast<int64_t>((pl.num_kg + 3) / 4) * (pl.sfa_blocks + pl.sfb_blocks) * 4;
  int64_t blocks = (warps + 7) / 8;
  if (blocks > 16 * static_cast<int64_t>(ctx->num_sms)) blocks = 16 * ctx->num_sms;
  sf_repack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(sa, sb, K / 32, pl.num_kg);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);

  CUtensorMap tA, tB, tSA, tSB;
  int rc = make_tensor_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, K, M, lda, 128, 128,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, K, N, ldb, 128,
                          pair && mcast ? 256 / g / 2 : 256 / g, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tSA, CU_TENSOR_MAP_DATA_TYPE_UINT32, img_a, 128,
                          static_cast<uint64_t>(pl.num_kg) * pl.sfa_blocks, 512, 128, 1,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tSB, CU_TENSOR_MAP_DATA_TYPE_UINT32, img_b, 128,
                          static_cast<uint64_t>(pl.num_kg) * pl.sfb_blocks, 512, 128, 2,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != TG_OK) return rc;

  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.num_m_tiles = pl.num_m_tiles;
  a.num_n_tiles = pl.num_n_tiles;
  a.num_k_blocks = pl.num_kg;
  a.D = D;
  a.ldd = ldd;
  a.epi = epi;
  a.sfa_blocks = pl.sfa_blocks;
  a.sfb_blocks = pl.sfb_blocks;
  a.raster_group = kRasterGroup;
  a.status = ctx->status;
  a.timeout_ns = wait_timeout_ns();
  const bool bf16_out = d_dtype == TG_D_BF16;
  if (!pair)
    return bf16_out ? launch_gemm_cfg<CfgMxBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                    : launch_gemm_cfg<CfgMxF32>(tA, tB, tSA, tSB, a, stream, ctx);
  if (mcast)
    return bf16_out ? launch_gemm_cfg<CfgMxPairMcBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                    : launch_gemm_cfg<CfgMxPairMcF32>(tA, tB, tSA, tSB, a, stream, ctx);
  return bf16_out ? launch_gemm_cfg<CfgMxPairBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                  : launch_gemm_cfg<CfgMxPairF32>(tA, tB, tSA, tSB, a, stream, ctx);
}

}  // namespace tg
