// Kernel configurations of the block-scaled FP4 GEMMs (packed E2M1 operands,
// .kind::mxf4nvf4): MXFP4 (.scale_vec::2X, E8M0 per 32 K) and NVFP4
// (.scale_vec::4X, UE4M3 per 16 K).  The plan, the scale rearrangement and
// the tensor maps are shared with MXFP8 (gemm_blockscaled.cu).
//
// A stage is 128 bytes = 256 packed values of K per row, four K64 MMAs.  Per
// stage a 128-row block needs 2 (MXFP4) or 4 (NVFP4) scale images, i.e. 24 or
// 48 TMEM columns with a 256-wide B tile; next to the 256-column accumulator
// that allows 6 (MXFP4) or 5 (NVFP4) pair stages within 512 columns.
#include "gemm_launch.cuh"

namespace tg {

namespace {
using CfgMxf4F32 = GemmCfg<1, kKindMxf4, 256, 1, 4, false>;
using CfgMxf4Bf16 = GemmCfg<1, kKindMxf4, 256, 1, 4, true>;
using CfgMxf4PairF32 = GemmCfg<2, kKindMxf4, 256, 1, 6, false>;
using CfgMxf4PairBf16 = GemmCfg<2, kKindMxf4, 256, 1, 6, true>;
using CfgNvf4F32 = GemmCfg<1, kKindNvf4, 256, 1, 4, false>;
using CfgNvf4Bf16 = GemmCfg<1, kKindNvf4, 256, 1, 4, true>;
using CfgNvf4PairF32 = GemmCfg<2, kKindNvf4, 256, 1, 5, false>;
using CfgNvf4PairBf16 = GemmCfg<2, kKindNvf4, 256, 1, 5, true>;
}  // namespace

int launch_gemm_fp4_cfg(int kind, bool pair, bool bf16_out, const CUtensorMap& tA,
                        const CUtensorMap& tB, const CUtensorMap& tSA, const CUtensorMap& tSB,
                        const GemmArgs& a, cudaStream_t stream, DeviceCtx* ctx) {
  if (kind == kKindMxf4) {
    if (!pair)
      return bf16_out ? launch_gemm_cfg<CfgMxf4Bf16>(tA, tB, tSA, tSB, a, stream, ctx)
                      : launch_gemm_cfg<CfgMxf4F32>(tA, tB, tSA, tSB, a, stream, ctx);
    return bf16_out ? launch_gemm_cfg<CfgMxf4PairBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                    : launch_gemm_cfg<CfgMxf4PairF32>(tA, tB, tSA, tSB, a, stream, ctx);
  }
  if (kind == kKindNvf4) {
    if (!pair)
      return bf16_out ? launch_gemm_cfg<CfgNvf4Bf16>(tA, tB, tSA, tSB, a, stream, ctx)
                      : launch_gemm_cfg<CfgNvf4F32>(tA, tB, tSA, tSB, a, stream, ctx);
    return bf16_out ? launch_gemm_cfg<CfgNvf4PairBf16>(tA, tB, tSA, tSB, a, stream, ctx)
                    : launch_gemm_cfg<CfgNvf4PairF32>(tA, tB, tSA, tSB, a, stream, ctx);
  }
  return TG_ERR_UNSUPPORTED;
}

}  // namespace tg
