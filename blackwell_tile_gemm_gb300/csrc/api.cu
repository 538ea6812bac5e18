// C entry points of libtgemm.so: argument checks, per-device state, the
// device status record, tensor-map encoding and the MXFP8 workspace.
//
// Every check happens before any launch, following the pages' rule that a
// contract violation is rejected rather than repaired ("Explicit CUDA tile
// patterns", section "Group, repeat, and atom axes": a failed contract is an
// error, never a search for another layout; "cp.async.bulk.tensor", section
// "Legality conditions": 16-byte aligned bases and outer byte strides).
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <unordered_map>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/tgemm.h"
#include "tg_internal.h"

namespace tg {

// Status record of each device: [0] code, [1] wait site, [2] block, [3] thread.
__device__ uint32_t g_status_record[4];
// SM clock readout of the GEMM kernels: per kind (dense bf16, MXFP8, MXFP4,
// NVFP4), the SM cycles, nanoseconds and MMA units summed over the launches
// made while tg_kernel_clock_record is on.
__device__ unsigned long long g_kernel_clock[4][3];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceCtx g_ctx[kMaxDevices];
uint64_t g_timeout_ns = 2000000000ull;
thread_local int t_last_cuda_error = 0;

// Library-owned device memory of one (device, stream): calls on different
// streams never share it, and calls on one stream are ordered.
//   ws        the workspace (scale images, re-pitched or gathered rows, the
//             skinny call's partial sums), grown on demand unless reserved;
//   partials, counters  the tail split's partial tiles and arrival counters;
//   reserved  set by tg_reserve_workspace: from then on no call on this
//             stream allocates or synchronises; a call that would need more
//             workspace returns TG_ERR_WORKSPACE instead.
struct StreamState {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  float* partials = nullptr;
  uint32_t* counters = nullptr;
  bool reserved = false;
};
std::map<std::pair<int, uintptr_t>, StreamState> g_streams;
// Device allocations the library has made (workspace, tail scratch).
uint64_t g_alloc_count = 0;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return TG_ERR_CUDA;
}

uint64_t wait_timeout_ns() {
  std::lock_guard<std::mutex> lk(g_mutex);
  return g_timeout_ns;
}

DeviceCtx* current_ctx() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    cuda_fail(cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mutex);
  DeviceCtx& c = g_ctx[dev];
  if (c.device == dev) return &c;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  void* st = nullptr;
  e = cudaGetSymbolAddress(&st, g_status_record);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  void* clk = nullptr;
  e = cudaGetSymbolAddress(&clk, g_kernel_clock);
  if (e != cudaSuccess) {
    cuda_fail(e);
    return nullptr;
  }
  c.num_sms = sms;
  c.status = static_cast<uint32_t*>(st);
  c.clock_acc = static_cast<unsigned long long*>(clk);
  c.device = dev;
  return &c;
}

namespace {
// Encoded maps by their complete input: an encoding is a pure function of
// these fields, so a hit returns exactly what a fresh encode would.  Bounded
// (cleared when full); keeps repeated calls on the same buffers off the
// driver's encoder.
struct MapKey {
  uint64_t base, inner, outer, row_bytes;
  uint32_t dtype, box_inner, box_outer, swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && inner == o.inner && outer == o.outer && row_bytes == o.row_bytes &&
           dtype == o.dtype && box_inner == o.box_inner && box_outer == o.box_outer &&
           swizzle == o.swizzle;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = 1469598103934665603ull;
    const uint64_t v[8] = {k.base, k.inner, k.outer, k.row_bytes, k.dtype, k.box_inner,
                           k.box_outer, k.swizzle};
    for (uint64_t x : v) h = (h ^ x) * 1099511628211ull;
    return static_cast<size_t>(h);
  }
};
constexpr size_t kMapCacheMax = 1024;
std::mutex g_map_mutex;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;
}  // namespace

int make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                       uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                       uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  // A zero extent is not encodable; callers never launch for empty problems,
  // but keep a valid map (extent 1) for unused descriptor parameters.
  if (inner == 0) inner = 1;
  if (outer == 0) outer = 1;
  const MapKey key{reinterpret_cast<uint64_t>(base), inner, outer, row_bytes,
                   static_cast<uint32_t>(dtype), box_inner, box_outer,
                   static_cast<uint32_t>(swizzle)};
  {
    std::lock_guard<std::mutex> lk(g_map_mutex);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *map = it->second;
      return TG_OK;
    }
  }
  {
    std::lock_guard<std::mutex> lk(g_mutex);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      cudaError_t e =
          cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess) return cuda_fail(e);
      if (q != cudaDriverEntryPointSuccess || fn == nullptr)
        return cuda_fail(cudaErrorSymbolNotFound);
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  std::lock_guard<std::mutex> lk(g_map_mutex);
  if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
  g_map_cache.emplace(key, *map);
  return TG_OK;
}

namespace {

std::pair<int, uintptr_t> stream_key(int dev, cudaStream_t stream) {
  return std::make_pair(dev, reinterpret_cast<uintptr_t>(stream));
}

// True when `stream` is being captured into a graph, or when its capture
// state cannot be read (the legacy stream while another stream captures):
// an allocation or a synchronisation then would break the capture.
bool stream_capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &st) != cudaSuccess) {
    cudaGetLastError();
    return true;
  }
  return st != cudaStreamCaptureStatusNone;
}

// Allocates the tail scratch of `t` (zeroed counters, ordered on `stream`).
// Caller holds g_mutex.
bool alloc_tail_scratch(StreamState& t, cudaStream_t stream) {
  float* part = nullptr;
  uint32_t* cnt = nullptr;
  if (cudaMalloc(&part, kTailPartialBytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  ++g_alloc_count;
  if (cudaMalloc(&cnt, kTailFlagWords * sizeof(uint32_t)) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(part);
    return false;
  }
  ++g_alloc_count;
  if (cudaMemsetAsync(cnt, 0, kTailFlagWords * sizeof(uint32_t), stream) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(part);
    cudaFree(cnt);
    return false;
  }
  t.partials = part;
  t.counters = cnt;
  return true;
}

// Grows the workspace of `t` to at least `bytes` (synchronising `stream`
// first when an older, smaller buffer may still be in use).  Caller holds
// g_mutex.
int grow_workspace(StreamState& t, size_t bytes, cudaStream_t stream) {
  if (t.ws) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaFree(t.ws);
    t.ws = nullptr;
    t.ws_bytes = 0;
  }
  const size_t want = bytes < (1u << 20) ? (1u << 20) : bytes;
  void* p = nullptr;
  cudaError_t e = cudaMalloc(&p, want);
  if (e != cudaSuccess) return cuda_fail(e);
  ++g_alloc_count;
  t.ws = p;
  t.ws_bytes = want;
  return TG_OK;
}

}  // namespace

bool tail_scratch(cudaStream_t stream, float** partials, uint32_t** counters) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lk(g_mutex);
  StreamState& t = g_streams[stream_key(dev, stream)];
  if (t.partials == nullptr) {
    // Without a reservation the scratch is allocated on first need, except
    // while the stream is captured (the product then runs unsplit).
    if (t.reserved || stream_capturing(stream) || !alloc_tail_scratch(t, stream)) return false;
  }
  *partials = t.partials;
  *counters = t.counters;
  return true;
}

void reset_tail_flags() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lk(g_mutex);
  for (auto& kv : g_streams)
    if (kv.first.first == dev && kv.second.counters)
      cudaMemset(kv.second.counters, 0, kTailFlagWords * sizeof(uint32_t));
}

void* device_workspace(size_t bytes, cudaStream_t stream, int* rc) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *rc = cuda_fail(e != cudaSuccess ? e : cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mutex);
  StreamState& t = g_streams[stream_key(dev, stream)];
  if (t.ws && t.ws_bytes >= bytes) return t.ws;
  if (t.reserved || stream_capturing(stream)) {
    *rc = TG_ERR_WORKSPACE;
    return nullptr;
  }
  *rc = grow_workspace(t, bytes, stream);
  return *rc == TG_OK ? t.ws : nullptr;
}

int reserve_workspace(cudaStream_t stream, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lk(g_mutex);
  if (stream_capturing(stream)) return TG_ERR_WORKSPACE;
  StreamState& t = g_streams[stream_key(dev, stream)];
  if (!t.ws || t.ws_bytes < bytes) {
    const int rc = grow_workspace(t, bytes, stream);
    if (rc != TG_OK) return rc;
  }
  if (t.partials == nullptr && !alloc_tail_scratch(t, stream)) return cuda_fail(cudaErrorMemoryAllocation);
  // The counters' zeroing (and any earlier use of a replaced buffer) is
  // complete before the reservation is reported.
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  t.reserved = true;
  return TG_OK;
}

uint64_t alloc_count() {
  std::lock_guard<std::mutex> lk(g_mutex);
  return g_alloc_count;
}

bool device_local(const void* ptr, int dev) {
  if (ptr == nullptr) return false;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice && a.device == dev;
}

bool operands_local(const void* const* ptrs, int n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  for (int i = 0; i < n; ++i)
    if (!device_local(ptrs[i], dev)) return false;
  return true;
}

int launch_gemm(int kind, const void* A, int64_t lda, const void* B, int64_t ldb,
                const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb, void* D,
                int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype, const Epi& epi,
                unsigned flags, cudaStream_t stream, DeviceCtx* ctx) {
  if (K == 0) return launch_fill_epilogue(D, ldd, M, N, d_dtype, epi, stream);
  const bool pair = (flags & TG_FLAG_CTA_PAIR) != 0;
  const bool mcast_flag = (flags & TG_FLAG_MULTICAST) != 0;
  int rc = TG_OK;
  if (kind == kKindBf16) {
    const bool mcast = bf16_uses_multicast(A, B, M, N, K, pair, mcast_flag);
    const Bf16Repitch rp = bf16_repitch_plan(lda, ldb, M, N, K, pair && mcast);
    if (rp.bytes != 0) {
      void* ws = device_workspace(rp.bytes, stream, &rc);
      if (ws == nullptr) return rc;
      return launch_gemm_bf16_repitched(rp, A, lda, B, ldb, D, ldd, static_cast<int>(M),
                                        static_cast<int>(N), static_cast<int>(K), d_dtype, epi,
                                        pair, mcast, ws, stream, ctx);
    }
    return launch_gemm_bf16_impl(A, lda, B, ldb, D, ldd, static_cast<int>(M),
                                 static_cast<int>(N), static_cast<int>(K), d_dtype, epi, pair,
                                 mcast, stream, ctx);
  }
  // Block-scaled multicast clusters (MXFP8 pairs) load B by TMA multicast:
  // only over memory of the current device.
  const void* ops[4] = {A, B, SFA, SFB};
  const bool mcast = mcast_flag && operands_local(ops, 4);
  uint8_t* ws = static_cast<uint8_t*>(
      device_workspace(blockscaled_workspace_bytes(kind, M, N, K, pair), stream, &rc));
  if (ws == nullptr) return rc;
  return launch_gemm_blockscaled_impl(kind, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd,
                                      static_cast<int>(M), static_cast<int>(N),
                                      static_cast<int>(K), d_dtype, epi, pair, mcast, ws,
                                      stream, ctx);
}

int check_epilogue(const tg_epilogue* epi, Epi* out) {
  Epi e{kEpiNone, 0.0f, 0.0f, nullptr};
  if (epi != nullptr) {
    if (epi->op < kEpiNone || epi->op > kEpiAffine) return TG_ERR_INVALID_ARG;
    e.op = epi->op;
    e.alpha = epi->alpha;
    e.beta = epi->beta;
    if (epi_uses_bias(e.op)) {
      if (epi->bias == nullptr) return TG_ERR_INVALID_ARG;
      if (!aligned16(epi->bias)) return TG_ERR_MISALIGNED;
      e.bias = epi->bias;
    }
  }
  *out = e;
  return TG_OK;
}

}  // namespace tg

using namespace tg;

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

// a_esize: bytes per ld unit of A and B; k_per_unit: K elements per ld unit
// (2 for packed FP4, whose rows are K / 2 bytes).
int check_gemm_common(const void* A, int64_t lda, const void* B, int64_t ldb, void* D,
                      int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype, int epilogue,
                      unsigned flags, int a_esize, int k_per_unit = 1) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return TG_ERR_INVALID_ARG;
  if (d_dtype != TG_D_F32 && d_dtype != TG_D_BF16) return TG_ERR_INVALID_ARG;
  if (epilogue < TG_EPI_NONE || epilogue > TG_EPI_BIAS_COL_SILU) return TG_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(TG_FLAG_CTA_PAIR | TG_FLAG_MULTICAST))
    return TG_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return TG_OK;
  if (D == nullptr || ldd < N) return TG_ERR_INVALID_ARG;
  const int d_esize = d_dtype == TG_D_F32 ? 4 : 2;
  if (!aligned16(D) || (ldd * d_esize) % 16 != 0) return TG_ERR_MISALIGNED;
  if (K == 0) return TG_OK;
  if (A == nullptr || B == nullptr || lda * k_per_unit < K || ldb * k_per_unit < K)
    return TG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B)) return TG_ERR_MISALIGNED;
  if ((lda * a_esize) % 16 != 0 || (ldb * a_esize) % 16 != 0) return TG_ERR_MISALIGNED;
  return TG_OK;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

namespace tg {

// Argument checks of the block-scaled call, shared with the variant that
// takes its scratch from a static array (gemm_mxfp8_noalloc.cu).
int check_blockscaled_args(int kind, const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           int epilogue, unsigned flags) {
  if (kind != kKindMxf8 && kind != kKindMxf4 && kind != kKindNvf4) return TG_ERR_INVALID_ARG;
  const int block = scale_block_of(kind);
  if (K % block != 0) return TG_ERR_INVALID_ARG;
  // Block-scaled multicast clusters are made of CTA pairs, for MXFP8 only.
  if ((flags & TG_FLAG_MULTICAST) && !(flags & TG_FLAG_CTA_PAIR)) return TG_ERR_INVALID_ARG;
  if (kind != kKindMxf8 && (flags & TG_FLAG_MULTICAST)) return TG_ERR_UNSUPPORTED;
  int rc = check_gemm_common(A, lda, B, ldb, D, ldd, M, N, K, d_dtype, epilogue, flags, 1,
                             kind == kKindMxf8 ? 1 : 2);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  if (K > 0 && (SFA == nullptr || SFB == nullptr || ld_sfa < K / block || ld_sfb < K / block))
    return TG_ERR_INVALID_ARG;
  return TG_OK;
}

}  // namespace tg

extern "C" {

int gemm_bf16_ex(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
                 int64_t M, int64_t N, int64_t K, int d_dtype, const tg_epilogue* epi,
                 unsigned flags, void* cuda_stream) {
  Epi e;
  int rc = check_epilogue(epi, &e);
  if (rc != TG_OK) return rc;
  rc = check_gemm_common(A, lda, B, ldb, D, ldd, M, N, K, d_dtype, TG_EPI_NONE, flags, 2);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  return launch_gemm(kKindBf16, A, lda, B, ldb, nullptr, 0, nullptr, 0, D, ldd, M, N, K,
                     d_dtype, e, flags, as_stream(cuda_stream), ctx);
}

int gemm_bf16(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
              int64_t M, int64_t N, int64_t K, int d_dtype, int epilogue, float epi_scalar,
              unsigned flags, void* cuda_stream) {
  if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_ADD_SCALAR) return TG_ERR_INVALID_ARG;
  const tg_epilogue e{epilogue, epi_scalar, 0.0f, nullptr};
  return gemm_bf16_ex(A, lda, B, ldb, D, ldd, M, N, K, d_dtype, &e, flags, cuda_stream);
}

int gemm_mxfp8_blockscaled_ex(const void* A, int64_t lda, const void* B, int64_t ldb,
                              const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                              void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                              int d_dtype, const tg_epilogue* epi, unsigned flags,
                              void* cuda_stream) {
  Epi e;
  int rc = check_epilogue(epi, &e);
  if (rc != TG_OK) return rc;
  rc = check_mxfp8_args(A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K, d_dtype,
                        TG_EPI_NONE, flags);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  return launch_gemm(kKindMxf8, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K,
                     d_dtype, e, flags, as_stream(cuda_stream), ctx);
}

int gemm_mxfp8_blockscaled(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           int epilogue, float epi_scalar, unsigned flags, void* cuda_stream) {
  if (epilogue != TG_EPI_NONE && epilogue != TG_EPI_ADD_SCALAR) return TG_ERR_INVALID_ARG;
  const tg_epilogue e{epilogue, epi_scalar, 0.0f, nullptr};
  return gemm_mxfp8_blockscaled_ex(A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K,
                                   d_dtype, &e, flags, cuda_stream);
}

}  // extern "C"

namespace {

int gemm_fp4_common(int kind, const void* A, int64_t lda, const void* B, int64_t ldb,
                    const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb, void* D,
                    int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                    const tg_epilogue* epi, unsigned flags, void* cuda_stream) {
  Epi e;
  int rc = check_epilogue(epi, &e);
  if (rc != TG_OK) return rc;
  rc = check_blockscaled_args(kind, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K,
                              d_dtype, TG_EPI_NONE, flags);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  return launch_gemm(kind, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K, d_dtype, e,
                     flags, as_stream(cuda_stream), ctx);
}

}  // namespace

extern "C" {

int gemm_bf16_skinny(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
                     int64_t M, int64_t N, int64_t K, int d_dtype, const tg_epilogue* epi,
                     int split_k, void* cuda_stream) {
  Epi e;
  int rc = check_epilogue(epi, &e);
  if (rc != TG_OK) return rc;
  if (split_k < 0) return TG_ERR_INVALID_ARG;
  rc = check_gemm_common(A, lda, B, ldb, D, ldd, M, N, K, d_dtype, TG_EPI_NONE, 0, 2);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  if (M > 128) return TG_ERR_UNSUPPORTED;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  cudaStream_t stream = as_stream(cuda_stream);
  if (K == 0) return launch_fill_epilogue(D, ldd, M, N, d_dtype, e, stream);
  float* ws = nullptr;
  const size_t ws_bytes = skinny_workspace_bytes(M, N, d_dtype, e.op);
  if (ws_bytes) {
    ws = static_cast<float*>(device_workspace(ws_bytes, stream, &rc));
    if (ws == nullptr) return rc;
  }
  return launch_gemm_skinny_impl(A, lda, B, ldb, D, ldd, static_cast<int>(M), static_cast<int>(N),
                                 static_cast<int>(K), d_dtype, e, split_k, ws, stream, ctx);
}

int gemm_bf16_gather(const void* A, int64_t lda, int64_t a_rows, const int32_t* row_idx,
                     int64_t M, const void* B, int64_t ldb, void* D, int64_t ldd, int64_t N,
                     int64_t K, int d_dtype, const tg_epilogue* epi, unsigned flags,
                     void* cuda_stream) {
  Epi e;
  int rc = check_epilogue(epi, &e);
  if (rc != TG_OK) return rc;
  if (flags & TG_FLAG_MULTICAST) return TG_ERR_UNSUPPORTED;
  if (flags & ~static_cast<unsigned>(TG_FLAG_CTA_PAIR | TG_FLAG_GATHER_TMA))
    return TG_ERR_UNSUPPORTED;
  if (a_rows < 0 || a_rows > kMaxDim) return TG_ERR_INVALID_ARG;
  // A is checked as an [a_rows, K] operand, D as [M, N].
  rc = check_gemm_common(A, lda, B, ldb, D, ldd, M, N, K, d_dtype, TG_EPI_NONE,
                         flags & TG_FLAG_CTA_PAIR, 2);
  if (rc != TG_OK || M == 0 || N == 0) return rc;
  if (K > 0 && (row_idx == nullptr || a_rows == 0)) return TG_ERR_INVALID_ARG;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  cudaStream_t stream = as_stream(cuda_stream);
  if (K == 0) return launch_fill_epilogue(D, ldd, M, N, d_dtype, e, stream);
  const bool pair = (flags & TG_FLAG_CTA_PAIR) != 0;
  if (flags & TG_FLAG_GATHER_TMA)
    return launch_gemm_bf16_gather_impl(A, lda, static_cast<int>(a_rows), row_idx,
                                        static_cast<int>(M), B, ldb, D, ldd, static_cast<int>(N),
                                        static_cast<int>(K), d_dtype, e, pair, stream, ctx);
  void* ws = device_workspace(gather_workspace_bytes(M, K), stream, &rc);
  if (ws == nullptr) return rc;
  return launch_gemm_bf16_pregather_impl(A, lda, static_cast<int>(a_rows), row_idx,
                                         static_cast<int>(M), B, ldb, D, ldd, static_cast<int>(N),
                                         static_cast<int>(K), d_dtype, e, pair, ws, stream, ctx);
}

int tg_gemm_tail_split(int64_t M, int64_t N, int64_t K, unsigned flags) {
  if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return -TG_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(TG_FLAG_CTA_PAIR)) return -TG_ERR_UNSUPPORTED;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return -TG_ERR_CUDA;
  return bf16_tail_split(M, N, K, (flags & TG_FLAG_CTA_PAIR) != 0, ctx);
}

int tg_gemm_multicast(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                      unsigned flags) {
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return -TG_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(TG_FLAG_CTA_PAIR | TG_FLAG_MULTICAST))
    return -TG_ERR_UNSUPPORTED;
  if (M == 0 || N == 0 || K == 0) return 0;   // nothing, or the K = 0 fill, runs
  return bf16_uses_multicast(A, B, M, N, K, (flags & TG_FLAG_CTA_PAIR) != 0,
                             (flags & TG_FLAG_MULTICAST) != 0)
             ? 1
             : 0;
}

int64_t tg_workspace_bytes(int call, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                           int d_dtype, int epi_op, unsigned flags) {
  if (M < 0 || N < 0 || K < 0 || lda < 0 || ldb < 0 || M > kMaxDim || N > kMaxDim ||
      K > kMaxDim)
    return -TG_ERR_INVALID_ARG;
  if (M == 0 || N == 0 || K == 0) return 0;
  const bool pair = (flags & TG_FLAG_CTA_PAIR) != 0;
  switch (call) {
    case TG_CALL_GEMM_BF16:
      // Multicast pair clusters take no copy, but fall back to plain pairs
      // (which may) for operands outside this device's memory: size for
      // the plain kernel.
      return static_cast<int64_t>(bf16_repitch_plan(lda, ldb, M, N, K, false).bytes);
    case TG_CALL_GEMM_MXFP8:
      if (K % 32) return -TG_ERR_INVALID_ARG;
      return static_cast<int64_t>(blockscaled_workspace_bytes(kKindMxf8, M, N, K, pair));
    case TG_CALL_GEMM_MXFP4:
      if (K % 32) return -TG_ERR_INVALID_ARG;
      return static_cast<int64_t>(blockscaled_workspace_bytes(kKindMxf4, M, N, K, pair));
    case TG_CALL_GEMM_NVFP4:
      if (K % 16) return -TG_ERR_INVALID_ARG;
      return static_cast<int64_t>(blockscaled_workspace_bytes(kKindNvf4, M, N, K, pair));
    case TG_CALL_GEMM_BF16_SKINNY:
      if (M > 128) return -TG_ERR_UNSUPPORTED;
      if (d_dtype != TG_D_F32 && d_dtype != TG_D_BF16) return -TG_ERR_INVALID_ARG;
      if (epi_op < kEpiNone || epi_op > kEpiAffine) return -TG_ERR_INVALID_ARG;
      return static_cast<int64_t>(skinny_workspace_bytes(M, N, d_dtype, epi_op));
    case TG_CALL_GEMM_BF16_GATHER:
      return (flags & TG_FLAG_GATHER_TMA) ? 0 : static_cast<int64_t>(gather_workspace_bytes(M, K));
    default:
      return -TG_ERR_INVALID_ARG;
  }
}

int tg_reserve_workspace(void* cuda_stream, int64_t bytes) {
  if (bytes < 0) return TG_ERR_INVALID_ARG;
  return reserve_workspace(as_stream(cuda_stream), static_cast<size_t>(bytes));
}

uint64_t tg_workspace_alloc_count(void) { return alloc_count(); }

int tg_gemm_repitch(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, unsigned flags) {
  if (M < 0 || N < 0 || K < 0 || lda < 0 || ldb < 0) return -TG_ERR_INVALID_ARG;
  if (flags & ~static_cast<unsigned>(TG_FLAG_CTA_PAIR | TG_FLAG_MULTICAST))
    return -TG_ERR_INVALID_ARG;
  const bool pair_clusters = (flags & TG_FLAG_CTA_PAIR) && (flags & TG_FLAG_MULTICAST);
  const Bf16Repitch rp = bf16_repitch_plan(lda, ldb, M, N, K, pair_clusters);
  return (rp.a ? 1 : 0) | (rp.b ? 2 : 0);
}

int tg_skinny_split_count(int64_t N, int64_t K, int split_k) {
  if (N < 1 || K < 1 || split_k < 0 || N > kMaxDim || K > kMaxDim) return -TG_ERR_INVALID_ARG;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return -TG_ERR_CUDA;
  int per = 0;
  return skinny_splits(N, K, split_k, ctx->num_sms, &per);
}

int gemm_mxfp4_blockscaled(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           const tg_epilogue* epi, unsigned flags, void* cuda_stream) {
  return gemm_fp4_common(kKindMxf4, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K,
                         d_dtype, epi, flags, cuda_stream);
}

int gemm_nvfp4_blockscaled(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           const tg_epilogue* epi, unsigned flags, void* cuda_stream) {
  return gemm_fp4_common(kKindNvf4, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M, N, K,
                         d_dtype, epi, flags, cuda_stream);
}

int tile_transpose_b16(const void* in, int64_t ld_in, void* out, int64_t ld_out, int64_t rows,
                       int64_t cols, void* cuda_stream) {
  if (rows < 0 || cols < 0 || rows > kMaxDim || cols > kMaxDim) return TG_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return TG_OK;
  if (in == nullptr || out == nullptr || ld_in < cols || ld_out < rows) return TG_ERR_INVALID_ARG;
  if (!aligned16(in) || !aligned16(out) || ld_in % 8 != 0 || ld_out % 8 != 0)
    return TG_ERR_MISALIGNED;
  // in spans [in, in + 2*((rows-1)*ld_in + cols)), out likewise: reject overlap.
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(in);
  const uintptr_t a1 = a0 + 2u * static_cast<uintptr_t>((rows - 1) * ld_in + cols);
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(out);
  const uintptr_t b1 = b0 + 2u * static_cast<uintptr_t>((cols - 1) * ld_out + rows);
  if (a0 < b1 && b0 < a1) return TG_ERR_INVALID_ARG;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  return launch_transpose_b16(in, ld_in, out, ld_out, rows, cols, as_stream(cuda_stream), ctx);
}

int tg_device_status(void* cuda_stream, uint32_t* site) {
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  cudaError_t e = cudaStreamSynchronize(as_stream(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e);
  uint32_t rec[4] = {0, 0, 0, 0};
  e = cudaMemcpyFromSymbol(rec, g_status_record, sizeof(rec));
  if (e != cudaSuccess) return cuda_fail(e);
  const uint32_t zero[4] = {0, 0, 0, 0};
  e = cudaMemcpyToSymbol(g_status_record, zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e);
  if (site) *site = rec[1];
  // A launch that gave up may have left tail-split flags set: start over.
  if (rec[0] != TG_OK) reset_tail_flags();
  return static_cast<int>(rec[0]);
}

int tg_kernel_clock_record(int enable) {
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  ctx->clock_on.store(false);
  // Launches already queued finish adding before the sums are read or cleared.
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  if (enable == 0) return TG_OK;
  const unsigned long long zero[4][3] = {};
  e = cudaMemcpyToSymbol(g_kernel_clock, zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e);
  ctx->clock_on.store(true);
  return TG_OK;
}

int tg_kernel_clock_read(int kind, double* mhz, uint64_t* units) {
  if (kind < TG_CLOCK_BF16 || kind > TG_CLOCK_NVFP4 || mhz == nullptr)
    return TG_ERR_INVALID_ARG;
  DeviceCtx* ctx = current_ctx();
  if (!ctx) return TG_ERR_CUDA;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned long long v[3] = {0, 0, 0};
  e = cudaMemcpyFromSymbol(v, g_kernel_clock, sizeof(v), sizeof(v) * static_cast<size_t>(kind));
  if (e != cudaSuccess) return cuda_fail(e);
  *mhz = v[1] ? static_cast<double>(v[0]) * 1e3 / static_cast<double>(v[1]) : 0.0;
  if (units) *units = v[2];
  return TG_OK;
}

int tg_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return TG_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mutex);
  g_timeout_ns = ns;
  return TG_OK;
}

const char* tg_status_string(int status) {
  switch (status) {
    case TG_OK: return "ok";
    case TG_ERR_INVALID_ARG: return "invalid argument";
    case TG_ERR_MISALIGNED: return "misaligned pointer or row stride";
    case TG_ERR_UNSUPPORTED: return "unsupported request";
    case TG_ERR_CUDA: return "CUDA error";
    case TG_ERR_TIMEOUT: return "device pipeline wait timed out";
    case TG_ERR_NO_SCRATCH: return "problem needs more scratch than the static no-allocation buffer";
    case TG_ERR_WORKSPACE:
      return "the stream's workspace is too small and may not grow now (reserved, or the stream is being captured)";
    default: return "unknown status";
  }
}

int tg_last_cuda_error(void) { return t_last_cuda_error; }

int tg_version(void) { return 200; }

}  // extern "C"
