// Block-scaled GEMMs: MXFP8 (.kind::mxf8f6f4 .scale_vec::1X, E4M3 with an
// E8M0 scale per 32 K), MXFP4 (.kind::mxf4nvf4 .scale_vec::2X, packed E2M1
// with an E8M0 scale per 32 K) and NVFP4 (.kind::mxf4nvf4 .scale_vec::4X,
// packed E2M1 with a UE4M3 scale per 16 K); f32 accumulation.
//
// Scale factors reach tensor memory as "tcgen05.mma" (section
// "Weight-stationary and block scaling") lays them out: scale row r sits in
// TMEM lane r % 32, byte column 4 * (r / 32) + sf, replicated in the four
// 32-lane slabs; the scale-factor id in the instruction descriptor is the
// byte at which an MMA's scale vector starts.  tcgen05.cp .32x128b.warpx4
// ("Explicit CUDA tile patterns", section "TMEM transfers": warpx4 adds four
// replicas 32 lanes apart) copies 32 rows of 16 bytes, so one shared-memory
// image of 128 scale rows x 4 consecutive scales is 512 bytes with byte
// (16 * l + 4 * j + t) = scale t of row 32 * j + l.
//
// A stage holds 128 bytes of K per row: 4 MMAs of 32 bytes, each reading
// V = 1, 2 or 4 scales per row (the .scale_vec width), i.e. V images per
// 128-row block and stage.  sf_repack_kernel writes those images from the
// caller's natural [rows, K / block] byte arrays into the workspace, ordered
// [stage][128-row block][image]; the GEMM fetches a stage's images of one
// operand with one TMA box.
//
// MXFP8 configurations live here, the FP4 ones in gemm_fp4.cu.  Single CTA:
// 128 x 256 tiles, 4 stages, one 256-column accumulator plus the scale
// columns of every stage; CTA pair: 256 x 256 tiles, 6 stages per CTA
// (NVFP4: 5, whose scale columns would not fit a sixth).
#include "gemm_launch.cuh"

namespace tg {

namespace {

using CfgMxF32 = GemmCfg<1, kKindMxf8, 256, 1, 4, false>;
using CfgMxBf16 = GemmCfg<1, kKindMxf8, 256, 1, 4, true>;
using CfgMxPairF32 = GemmCfg<2, kKindMxf8, 256, 1, 6, false>;
using CfgMxPairBf16 = GemmCfg<2, kKindMxf8, 256, 1, 6, true>;
using CfgMxPairMcF32 = GemmCfg<2, kKindMxf8, 256, 1, 6, false, true>;
using CfgMxPairMcBf16 = GemmCfg<2, kKindMxf8, 256, 1, 6, true, true>;

struct SfImage {
  const uint8_t* src;   // [rows, kblocks] bytes, row stride ld
  int64_t ld;
  int rows;
  int blocks;           // 128-row blocks per stage in the image
  uint32_t* dst;        // [num_kg / groups][blocks][groups][128] words
  int vec16;            // src and ld are 16-byte aligned: whole chunks load as uint4
};

// Scale group g (scales 4g .. 4g+3 of each row) belongs to stage g / groups
// as image g % groups.  Image word (4*l + j) of 128-row block b holds the
// scales of row 128*b + 32*j + l (low byte first); rows or scales past the
// end are zero.  Work unit: one warp per (image, block,
// quad of K groups, l-octet).  Lane (4*l' + j) reads the 16 scale bytes of
// K groups 4*quad .. 4*quad+3 of its row and writes one word into each of
// those four images, so that each warp store covers 32 consecutive words
// (128 bytes) of one image.
__global__ void sf_repack_kernel(SfImage a, SfImage b, int kblocks, int num_kg, int groups) {
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
      const uint8_t* src = s.src + static_cast<int64_t>(row) * s.ld + 16 * quad;
      if (16 * quad + 16 <= kblocks && s.vec16) {
        // The 16 scales of this quad are a 16-byte aligned chunk of the row.
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(src));
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
      } else {
#pragma unroll
        for (int t = 0; t < 16; ++t)
          if (16 * quad + t < kblocks)
            v[t >> 2] |= static_cast<uint32_t>(__ldg(src + t)) << (8 * (t & 3));
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kg = 4 * quad + t;
      if (kg < num_kg) {
        const int64_t img =
            (static_cast<int64_t>(kg / groups) * s.blocks + blk) * groups + kg % groups;
        s.dst[img * 128 + 4 * l + j] = v[t];
      }
    }
  }
}

struct BsPlan {
  int num_m_tiles, num_n_tiles;
  int num_stages;   // stages of 128 bytes of K per row
  int groups;       // scale images per 128-row block and stage
  int num_kg;       // groups of 4 scales per row, padded to whole stages
  int kblocks;      // scales per row
  int sfa_blocks, sfb_blocks;
};

BsPlan plan_bs(int kind, int64_t M, int64_t N, int64_t K, bool pair) {
  const int g = pair ? 2 : 1;
  BsPlan p{};
  p.num_m_tiles = ceil_div_i(M, 128 * g);
  p.num_n_tiles = ceil_div_i(N, 256);
  p.num_stages = ceil_div_i(K, stage_k_of(kind));
  p.groups = scale_vec_of(kind);
  p.num_kg = p.num_stages * p.groups;
  p.kblocks = static_cast<int>(K / scale_block_of(kind));
  p.sfa_blocks = p.num_m_tiles * g;
  p.sfb_blocks = p.num_n_tiles * 2;
  return p;
}

}  // namespace

size_t blockscaled_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K, bool pair) {
  const BsPlan p = plan_bs(kind, M, N, K, pair);
  return static_cast<size_t>(p.sfa_blocks + p.sfb_blocks) * p.num_kg * 512u;
}

size_t mxfp8_workspace_bytes(int64_t M, int64_t N, int64_t K, bool pair) {
  return blockscaled_workspace_bytes(kKindMxf8, M, N, K, pair);
}

int launch_gemm_blockscaled_impl(int kind, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, const void* SFA, int64_t ld_sfa, const void* SFB,
                                 int64_t ld_sfb, void* D, int64_t ldd, int M, int N, int K,
                                 int d_dtype, const Epi& epi, bool pair, bool mcast,
                                 uint8_t* sf_workspace, cudaStream_t stream, DeviceCtx* ctx,
                                 bool no_scratch) {
  const BsPlan pl = plan_bs(kind, M, N, K, pair);
  const int g = pair ? 2 : 1;
  uint8_t* img_a = sf_workspace;
  uint8_t* img_b = sf_workspace + static_cast<size_t>(pl.sfa_blocks) * pl.num_kg * 512u;

  auto vec16 = [](const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) % 16 == 0 && ld % 16 == 0) ? 1 : 0;
  };
  SfImage sa{static_cast<const uint8_t*>(SFA), ld_sfa, M, pl.sfa_blocks,
             reinterpret_cast<uint32_t*>(img_a), vec16(SFA, ld_sfa)};
  SfImage sb{static_cast<const uint8_t*>(SFB), ld_sfb, N, pl.sfb_blocks,
             reinterpret_cast<uint32_t*>(img_b), vec16(SFB, ld_sfb)};
  const int64_t warps =
      static_cast<int64_t>((pl.num_kg + 3) / 4) * (pl.sfa_blocks + pl.sfb_blocks) * 4;
  int64_t blocks = (warps + 7) / 8;
  if (blocks > 16 * static_cast<int64_t>(ctx->num_sms)) blocks = 16 * ctx->num_sms;
  sf_repack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(sa, sb, pl.kblocks,
                                                                       pl.num_kg, pl.groups);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);

  // Operand rows are bytes: one E4M3 or two packed E2M1 values per byte.
  const uint64_t row_bytes = kind == kKindMxf8 ? static_cast<uint64_t>(K)
                                               : static_cast<uint64_t>(K) / 2;
  CUtensorMap tA, tB, tSA, tSB;
  int rc = make_tensor_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, M, lda, 128, 128,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, N, ldb, 128,
                          pair && mcast ? 256 / g / 2 : 256 / g, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  // Scale images: one box row = one 128-row block's `groups` images of a
  // stage (64-bit elements keep the box within 256 elements).
  const uint32_t img_elems = static_cast<uint32_t>(pl.groups) * 64;
  rc = make_tensor_map_2d(&tSA, CU_TENSOR_MAP_DATA_TYPE_UINT64, img_a, img_elems,
                          static_cast<uint64_t>(pl.num_stages) * pl.sfa_blocks,
                          static_cast<uint64_t>(img_elems) * 8, img_elems, 1,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tSB, CU_TENSOR_MAP_DATA_TYPE_UINT64, img_b, img_elems,
                          static_cast<uint64_t>(pl.num_stages) * pl.sfb_blocks,
                          static_cast<uint64_t>(img_elems) * 8, img_elems, 2,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != TG_OK) return rc;

  GemmArgs a{};
  a.M = M;
  a.N = N;
  a.K = K;
  a.num_m_tiles = pl.num_m_tiles;
  a.num_n_tiles = pl.num_n_tiles;
  a.num_k_blocks = pl.num_stages;
  a.D = D;
  a.ldd = ldd;
  a.epi = epi;
  a.sfa_blocks = pl.sfa_blocks;
  a.sfb_blocks = pl.sfb_blocks;
  a.status = ctx->status;
  a.timeout_ns = wait_timeout_ns();
  a.no_scratch = no_scratch;
  const bool bf16_out = d_dtype == TG_D_BF16;
  if (kind != kKindMxf8)
    return launch_gemm_fp4_cfg(kind, pair, bf16_out, tA, tB, tSA, tSB, a, stream, ctx);
  if (!pair)
    return bf16_out ? launch_gemm_cfg<CfgMxBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                    : launch_gemm_cfg<CfgMxF32>(tA, tB, tSA, tSB, a, stream, ctx);
  if (mcast)
    return bf16_out ? launch_gemm_cfg<CfgMxPairMcBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                    : launch_gemm_cfg<CfgMxPairMcF32>(tA, tB, tSA, tSB, a, stream, ctx);
  return bf16_out ? launch_gemm_cfg<CfgMxPairBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                  : launch_gemm_cfg<CfgMxPairF32>(tA, tB, tSA, tSB, a, stream, ctx);
}

int launch_gemm_mxfp8_impl(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int M, int N, int K, int d_dtype,
                           const Epi& epi, bool pair, bool mcast, uint8_t* sf_workspace,
                           cudaStream_t stream, DeviceCtx* ctx, bool no_scratch) {
  return launch_gemm_blockscaled_impl(kKindMxf8, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D,
                                      ldd, M, N, K, d_dtype, epi, pair, mcast, sf_workspace,
                                      stream, ctx, no_scratch);
}

}  // namespace tg
