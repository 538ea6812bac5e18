// Host launch of gemm_tcgen05_kernel<Cfg>: grid sizing, cluster attribute,
// dynamic shared memory opt-in (once per device and configuration).
#pragma once

#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_kernel.cuh"
#include "tg_internal.h"

namespace tg {

template <class C>
struct LaunchState {
  // Per device: 0 = not prepared, otherwise 1 + max co-resident CTA units.
  static inline std::atomic<int> units[64];
};

template <class C>
int gemm_units_for_device(DeviceCtx* ctx) {
  std::atomic<int>& slot = LaunchState<C>::units[ctx->device];
  int u = slot.load(std::memory_order_acquire);
  if (u > 0) return u - 1;
  auto kern = gemm_tcgen05_kernel<C>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return -cuda_fail(e);
  int units = ctx->num_sms / C::kClusterCtas;
  if constexpr (C::kClusterCtas > 1) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(C::kClusterCtas * units), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
    if (e != cudaSuccess) return -cuda_fail(e);
    if (clusters > 0 && clusters < units) units = clusters;
  }
  if (units < 1) units = 1;
  slot.store(units + 1, std::memory_order_release);
  return units;
}

// Tail split of `num_tiles` tiles over `units_max` units (see GemmArgs):
// returns S (1: none) and sets W (full waves) and R (tiles left over).
template <class C>
int tail_split_for(int num_tiles, int num_k_blocks, int units_max, int* W, int* R) {
  *W = num_tiles / units_max;
  *R = num_tiles - *W * units_max;
  // Measured on GB300 (graph-replayed, per call): a split K over otherwise
  // idle units pays off for dense bf16 when the last wave's tiles fill at
  // most half of the units (512 x 512 x 8192: 43 -> 30 us; 1024 x 1024 x
  // 8192 in pairs: 45 -> 39 us; after full waves 4096^3 93.5 -> 90.4 us,
  // 8192^3 in pairs 654 -> 640 us).  For the block-scaled kinds the exchange
  // of partial tiles cost more than it saved (1024 x 1024 x 8192 MXFP8:
  // 29 -> 33 us).  So: dense kinds only, and only the configurations whose
  // epilogue does the exchange (two accumulators, box-wise TMA stores).
  if (C::kMcast || C::kMx || !C::kTmaStore || C::kAccBufs != 2) return 1;
  if (*R == 0 || 2 * *R > units_max) return 1;
  int S = units_max / *R;
  if (S > 4) S = 4;
  while (S >= 2 && num_k_blocks < 4 * S) --S;
  // Every piece publishes its partial tile; one counter per epilogue warp.
  const size_t bytes = static_cast<size_t>(*R) * S * C::kCtaGroup * 128 * C::BN * 4;
  if (S < 2 || bytes > kTailPartialBytes || *R * C::kCtaGroup * C::kEpiWarps > kTailFlagWords)
    return 1;
  return S;
}

template <class C>
int launch_gemm_cfg(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tSFA,
                    const CUtensorMap& tSFB, const GemmArgs& args, cudaStream_t stream,
                    DeviceCtx* ctx) {
  const int units_max = gemm_units_for_device<C>(ctx);
  if (units_max < 0) return TG_ERR_CUDA;
  const int num_tiles = (args.num_m_tiles + C::kPairs - 1) / C::kPairs * args.num_n_tiles;
  int units = num_tiles < units_max ? num_tiles : units_max;
  GemmArgs a = args;
  // Tile order (measured on GB300, 8192^3 in pairs: bf16 0.583 -> 0.574 ms,
  // DRAM reads 1096 -> 885 MB a launch; MXFP8 0.333 -> 0.326 ms; 4096^3
  // single CTAs 0.094 -> 0.090 ms): bands of 4096 rows for CTA pairs and of
  // 384 rows for single CTAs, n walked backwards in every other band, K
  // backwards in every other wave.
  a.raster_group = (C::kCtaGroup == 2 ? 4096 : 384) / (128 * C::kCtaGroup * C::kPairs);
  if (a.raster_group < 1) a.raster_group = 1;
  a.n_snake = 1;
  a.k_snake = 1;
  a.full_tiles = num_tiles;
  a.tail_split = 1;
  a.tail_items = 0;
  a.partials = nullptr;
  a.counters = nullptr;
  a.clk = clock_slot(ctx, C::kKind);
  if (!args.no_scratch) {
    // Tail split: W full waves of whole tiles over all units; the R tiles of
    // a last, partial wave are cut into S K-pieces (S <= units / R, at most
    // 4, each piece at least 4 stages) so that R * S units finish together.
    // Calls that must not allocate (no_scratch) never split.
    int W = 0, R = 0;
    const int S = tail_split_for<C>(num_tiles, args.num_k_blocks, units_max, &W, &R);
    float* part = nullptr;
    uint32_t* counters = nullptr;
    if (S >= 2 && tail_scratch(stream, &part, &counters)) {
      a.full_tiles = W * units_max;
      a.tail_split = S;
      a.tail_items = R * S;
      a.partials = part;
      a.counters = counters;
      units = W > 0 ? units_max : R * S;
    }
  }
  // D for the TMA-store epilogue: [M rows][N columns] at row stride ldd,
  // boxes of 32 rows x 128 bytes (the API checks D's 16-byte alignment).
  CUtensorMap tD = tA;
  if constexpr (C::kTmaStore) {
    const int esize = C::kBf16Out ? 2 : 4;
    const int rc = make_tensor_map_2d(
        &tD, C::kBf16Out ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
        args.D, static_cast<uint64_t>(args.N), static_cast<uint64_t>(args.M),
        static_cast<uint64_t>(args.ldd) * esize, C::kStgRowBytes / esize, 32,
        C::kStgRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc != TG_OK) return rc;
  }
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(static_cast<unsigned>(units * C::kClusterCtas), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  // Programmatic dependent launch: the kernel's prologue may overlap the
  // previous kernel of the stream (the kernel waits before touching memory).
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (C::kClusterCtas > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C::kClusterCtas;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<C>, tA, tB, tSFA, tSFB, tD, a);
  if (e != cudaSuccess) return cuda_fail(e);
  return TG_OK;
}

inline int ceil_div_i(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// Launches the FP4 configuration of `kind` (kKindMxf4 / kKindNvf4) with the
// tensor maps and arguments the shared block-scaled plan built
// (gemm_fp4.cu).  Multicast clusters are not built for FP4.
int launch_gemm_fp4_cfg(int kind, bool pair, bool bf16_out, const CUtensorMap& tA,
                        const CUtensorMap& tB, const CUtensorMap& tSA, const CUtensorMap& tSB,
                        const GemmArgs& a, cudaStream_t stream, DeviceCtx* ctx);

}  // namespace tg
