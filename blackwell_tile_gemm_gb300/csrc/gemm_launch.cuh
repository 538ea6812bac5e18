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
  if constexpr (C::kCtaGroup == 2) {
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

template <class C>
int launch_gemm_cfg(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tSFA,
                    const CUtensorMap& tSFB, const GemmArgs& args, cudaStream_t stream,
                    DeviceCtx* ctx) {
  const int units_max = gemm_units_for_device<C>(ctx);
  if (units_max < 0) return TG_ERR_CUDA;
  const int num_tiles = (args.num_m_tiles + C::kPairs - 1) / C::kPairs * args.num_n_tiles;
  const int units = num_tiles < units_max ? num_tiles : units_max;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(units * C::kClusterCtas), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  if constexpr (C::kCtaGroup == 2) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C::kClusterCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tcgen05_kernel<C>, tA, tB, tSFA, tSFB, args);
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
