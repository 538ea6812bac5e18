// gemm_mxfp8_blockscaled_noalloc: the block-scaled MXFP8 GEMM for callers
// that must not allocate device memory.
//
// The regular entry point rearranges the scale factors into a workspace that
// the library allocates with cudaMalloc the first time a problem needs it.
// Some callers cannot allow that: a host framework that owns all device
// memory through its own pool (a raw cudaMalloc bypasses its accounting and
// can fail once the pool has reserved the device), a serving loop on a
// latency budget (cudaMalloc / cudaFree can synchronise the whole device), or
// a deployment that forbids any allocation after start-up.  This variant
// keeps its scratch in a fixed-size array that is part of the library's
// device image instead, so it never allocates.
//
// Properties a caller must know:
//   * The scratch is kNoAllocScratchBytes (8 MiB) per GPU, reserved on every
//     GPU that loads the library, for as long as the process lives.  A problem
//     needs (ceil(M/r)*r/128 + ceil(N/256)*2) * ceil(K/128) * 512 bytes, where
//     r = 256 with TG_FLAG_CTA_PAIR and 128 without (4 MiB at M=N=K=8192);
//     larger problems are rejected with TG_ERR_NO_SCRATCH before anything runs.
//   * All calls on a device share the one array.  Calls whose kernels can
//     overlap on the GPU (different streams without ordering between them)
//     race on it; order them, or use the regular entry point.
//   * The array keeps whatever the last call wrote.  Nothing needs clearing:
//     every call rewrites each scratch byte it later reads.
//   * The first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture begins.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/tgemm.h"
#include "tg_internal.h"

namespace tg {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t{8} << 20;
constexpr int kMaxDevicesNoAlloc = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
uint8_t* g_noalloc_addr[kMaxDevicesNoAlloc] = {};

// Device address of the scratch array on the current device (looked up once
// per device, with that device current).  nullptr on failure.
uint8_t* noalloc_scratch(int* rc) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    *rc = cuda_fail(e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevicesNoAlloc) {
    *rc = cuda_fail(cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_noalloc_mutex);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *rc = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return nullptr;
    }
    g_noalloc_addr[dev] = static_cast<uint8_t*>(p);
  }
  return g_noalloc_addr[dev];
}

}  // namespace
}  // namespace tg

using namespace tg;

extern "C" int gemm_mxfp8_blockscaled_noalloc(const void* A, int64_t lda, const void* B,
                                              int64_t ldb, const void* SFA, int64_t ld_sfa,
                                              const void* SFB, int64_t ld_sfb, void* D,
                                              int64_t ldd, int64_t M, int64_t N, int64_t K,
                                              int d_dtype, int epilogue, float epi_scalar,
                                              unsigned flags, void* cuda_stream) {
  if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_ADD_SCALAR) return TG_ERR_INVALID_ARG;
  int rc = check_mxfp8_args(A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K, d_dtype,
                            epilogue, flags);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  const Epi epi{epilogue, epi_scalar, 0.0f, nullptr};
  if (K == 0) return launch_fill_epilogue(D, ldd, M, N, d_dtype, epi, stream);
  const bool pair = (flags & TG_FLAG_CTA_PAIR) != 0;
  if (mxfp8_workspace_bytes(M, N, K, pair) > kNoAllocScratchBytes) return TG_ERR_NO_SCRATCH;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  uint8_t* scratch = noalloc_scratch(&rc);
  if (scratch == nullptr) return rc;
  // Multicast clusters only over operands in this device's memory.
  const void* ops[4] = {A, B, SFA, SFB};
  const bool mcast = (flags & TG_FLAG_MULTICAST) != 0 && operands_local(ops, 4);
  // no_scratch: the launcher must not turn on anything that allocates.
  return launch_gemm_mxfp8_impl(A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd,
                                static_cast<int>(M), static_cast<int>(N), static_cast<int>(K),
                                d_dtype, epi, pair, mcast, scratch, stream, ctx,
                                /*no_scratch=*/true);
}
