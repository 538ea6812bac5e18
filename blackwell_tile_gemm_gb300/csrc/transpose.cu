// tile_transpose_b16: out[j, i] = in[i, j] on raw 16-bit patterns.
//
// Built from the data-movement instructions of "ldmatrix / stmatrix" (TVM TIRx
// tile-operation guide): .trans transposes each 8x8 matrix of 16-bit
// elements (section "Transpose and stores": register element (row, 2w+h)
// comes from shared element (2w+h, row), owned by lane 4*row + w), and
// stmatrix writes a register image back to the rows its address providers
// name (lane 8*matrix + row supplies that row's address).  Tiles move with
// TMA ("cp.async.bulk.tensor": descriptor-defined boxes, loads completing on
// an mbarrier, stores as bulk groups; out-of-range elements of a load read
// zero and out-of-range elements of a store are not written).
//
// Persistent kernel, two CTAs per SM, each walking 64 x 64 tiles through a
// 4-stage ring:
//   1. one thread TMA-loads the input tile into stage s with 128-byte
//      swizzle: 16-byte chunk c of row r lands at chunk c ^ (r % 8), so the
//      8 rows an ldmatrix phase touches fall in 8 different bank groups;
//   2. each warp runs ldmatrix.x4.trans on S blocks (8w, 8c) and stmatrix.x4
//      into the output tile at block (8c, 8w), same swizzle;
//   3. one thread TMA-stores the output tile (edge tiles: element-wise stores
//      inside the array) and refills stage s.
#include <atomic>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "tg_internal.h"
#include "tg_ptx.cuh"

namespace tg {

namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;
constexpr int kStages = 4;
constexpr int kTileBytes = kTile * kTile * 2;     // 8 KB
constexpr int kSmemBytes = 2 * kStages * kTileBytes + 1024 + 64;
constexpr uint32_t kSiteTransposeFull = 20;

__device__ __forceinline__ uint32_t chunk_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads, 2)
    transpose_b16_kernel(const __grid_constant__ CUtensorMap tm_in,
                         const __grid_constant__ CUtensorMap tm_out, uint16_t* __restrict__ out,
                         int64_t ld_out, int rows, int cols, int tiles_r, int tiles_c,
                         uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* in_tiles = smem;                             // [kStages][8 KB]
  uint8_t* out_tiles = smem + kStages * kTileBytes;     // [kStages][8 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + 2 * kStages * kTileBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kStages);

  const int tid = threadIdx.x;
  const int num_tiles = tiles_r * tiles_c;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_in);
    prefetch_tensormap(&tm_out);
  }
  __syncthreads();
  // Programmatic dependent launch: the set-up above may overlap the end of
  // the previous kernel in the stream; global memory is touched only after
  // it has completed and its writes are visible.
  griddep_wait();
  const WaitGuard guard{status, abort_flag, timeout_ns};
  const uint64_t pol = policy_evict_first();

  auto issue_load = [&](int i, int s) {
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int ti = t / tiles_c, tj = t % tiles_c;
    mbar_arrive_expect_tx(&full[s], kTileBytes);
    tma_load_2d(smem_addr(in_tiles + s * kTileBytes), &tm_in, smem_addr(&full[s]), tj * kTile,
                ti * kTile, pol);
  };
  // This CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int my_tiles =
      num_tiles > static_cast<int>(blockIdx.x)
          ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
          : 0;
  if (tid == 0) {
    for (int i = 0; i < kStages && i < my_tiles; ++i) issue_load(i, i);
    // This CTA's last load is issued: the next kernel may launch.
    if (my_tiles <= kStages) griddep_launch_dependents();
  }

  const int w = tid >> 5, lane = tid & 31;
  const int m = lane >> 3, rr = lane & 7;
  bool ok = true;
  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % kStages;
    const uint32_t parity = static_cast<uint32_t>(i / kStages) & 1u;
    if (!mbar_try_wait(smem_addr(&full[s]), parity) &&
        !mbar_wait(&full[s], parity, guard, kSiteTransposeFull)) {
      ok = false;
    }
    // The store that last read out[s] (kStages tiles ago) must be done.
    if (tid == 0) bulk_wait_group_read<kStages - 1>();
    __syncthreads();
    if (!ok || *abort_flag) break;
    const uint32_t sS = smem_addr(in_tiles + s * kTileBytes);
    const uint32_t sT = smem_addr(out_tiles + s * kTileBytes);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ch = 4 * h + m;      // S block column = T block row
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(sS + chunk_offset(8 * w + rr, ch), r0, r1, r2, r3);
      stmatrix_x4(sT + chunk_offset(8 * ch + rr, w), r0, r1, r2, r3);
    }
    // Shared writes (stmatrix) and reads (ldmatrix) -> async proxy (TMA).
    fence_proxy_async_smem();
    __syncthreads();
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const int ti = t / tiles_c, tj = t % tiles_c;
    const bool full_tile = (ti + 1) * kTile <= rows && (tj + 1) * kTile <= cols;
    if (!full_tile) {
      // Edge tile: element-wise stores inside [cols, rows] only, so nothing
      // outside the caller's array (its row padding included) is written.
      const uint8_t* T = out_tiles + s * kTileBytes;
      for (int c = tid; c < kTile * 8; c += kThreads) {
        const int r = c >> 3, chunk = c & 7;
        const int oj = tj * kTile + r, oi = ti * kTile + chunk * 8;
        if (oj >= cols) continue;
        const uint4 x = *reinterpret_cast<const uint4*>(T + chunk_offset(r, chunk));
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
        uint16_t* dst = out + static_cast<int64_t>(oj) * ld_out;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (oi + e < rows) dst[oi + e] = static_cast<uint16_t>(w4[e >> 1] >> (16 * (e & 1)));
      }
      __syncthreads();     // out[s] is free again, in[s] was read above
    }
    if (tid == 0) {
      if (full_tile) {
        tma_store_2d(&tm_out, sT, ti * kTile, tj * kTile);
        bulk_commit_group();
      }
      if (i + kStages < my_tiles) issue_load(i + kStages, s);
      if (i + kStages == my_tiles - 1) griddep_launch_dependents();
    }
  }
  if (tid == 0) {
    bulk_wait_group0();
    if (!ok) {
      // Gave up: let loads already issued land before the CTA exits.
      for (int s = 0; s < kStages; ++s) mbar_wait_drain(&full[s], 0, timeout_ns);
    }
  }
}

}  // namespace

int launch_transpose_b16(const void* in, int64_t ld_in, void* out, int64_t ld_out, int64_t rows,
                         int64_t cols, cudaStream_t stream, DeviceCtx* ctx) {
  const int64_t tiles_r = (rows + kTile - 1) / kTile;
  const int64_t tiles_c = (cols + kTile - 1) / kTile;
  if (tiles_r * tiles_c > 0x7FFFFFFF) return TG_ERR_UNSUPPORTED;
  CUtensorMap tm_in, tm_out;
  int rc = make_tensor_map_2d(&tm_in, CU_TENSOR_MAP_DATA_TYPE_UINT16, in,
                              static_cast<uint64_t>(cols), static_cast<uint64_t>(rows),
                              static_cast<uint64_t>(ld_in) * 2, kTile, kTile,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tm_out, CU_TENSOR_MAP_DATA_TYPE_UINT16, out,
                          static_cast<uint64_t>(rows), static_cast<uint64_t>(cols),
                          static_cast<uint64_t>(ld_out) * 2, kTile, kTile,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  // Once per device (setting it twice is harmless; the flag is atomic so
  // that concurrent first calls do not race on it).
  static std::atomic<bool> attr_set[64];
  if (!attr_set[ctx->device].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(transpose_b16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    attr_set[ctx->device].store(true, std::memory_order_release);
  }
  const int64_t tiles = tiles_r * tiles_c;
  int64_t grid = 2 * static_cast<int64_t>(ctx->num_sms);
  if (grid > tiles) grid = tiles;
  // Programmatic dependent launch (the kernel waits before touching memory).
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, transpose_b16_kernel, tm_in, tm_out,
                                     static_cast<uint16_t*>(out), ld_out, static_cast<int>(rows),
                                     static_cast<int>(cols), static_cast<int>(tiles_r),
                                     static_cast<int>(tiles_c), ctx->status, wait_timeout_ns());
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

}  // namespace tg
