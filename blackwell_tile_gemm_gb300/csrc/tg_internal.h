// Host-side pieces shared by the translation units of libtgemm.so.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/tgemm.h"
#include "epilogue.cuh"
#include "gemm_kinds.h"

namespace tg {

// Per-device state, created on first use of a device.
struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  uint32_t* status = nullptr;      // device address of the 4-word status record
  // SM clock readout (tg_kernel_clock_record): device address of the
  // [kind][cycles, nanoseconds, units] sums, and whether launches add to it.
  unsigned long long* clock_acc = nullptr;
  std::atomic<bool> clock_on{false};
};

// Accumulator slot of GEMM kind `kind` (gemm_kinds.h) for the next launch, or
// nullptr while the clock readout is off.
inline unsigned long long* clock_slot(DeviceCtx* ctx, int kind) {
  return ctx->clock_on.load(std::memory_order_relaxed) ? ctx->clock_acc + 3 * kind : nullptr;
}

// Context of the current device (cudaGetDevice); nullptr on CUDA failure
// (the failure is recorded for tg_last_cuda_error).
DeviceCtx* current_ctx();

// Records a CUDA error for tg_last_cuda_error() and returns TG_ERR_CUDA.
int cuda_fail(cudaError_t e);

// Deadline of bounded device waits (ns).
uint64_t wait_timeout_ns();

// 2-D tiled tensor map over a row-major array: `inner` elements per row
// (contiguous), `outer` rows, `row_bytes` between rows.  Box = box_inner x
// box_outer elements.  Out-of-range box elements read zeros.
int make_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                       uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                       uint32_t box_outer, CUtensorMapSwizzle swizzle);

// Library-owned device workspace for (current device, `stream`), at least
// `bytes` long.  Without a reservation it is grown on demand (growing
// synchronises the stream first); a reserved workspace never grows.  When it
// is too small and cannot grow (reserved, or the stream is being captured)
// *rc = TG_ERR_WORKSPACE; on a CUDA failure *rc = TG_ERR_CUDA.  nullptr then.
void* device_workspace(size_t bytes, cudaStream_t stream, int* rc);

// tg_reserve_workspace: workspace of at least `bytes` plus the tail scratch
// for (current device, `stream`), allocated now; later calls on the stream
// neither allocate nor synchronise.
int reserve_workspace(cudaStream_t stream, size_t bytes);
// Device allocations made by the library so far.
uint64_t alloc_count();

// Scratch for the tail split of the persistent GEMM (partial tiles of the
// last wave's K pieces, and their arrival counters), one set per (device,
// stream) so that calls on different streams never share it.  Allocated by a
// reservation or on the first call that splits on that stream; the counters
// start at zero and every launch leaves them at zero.  false if it cannot be
// had (the call then runs without a split).
constexpr size_t kTailPartialBytes = size_t{20} << 20;   // >= 152 slots of 128 KiB
constexpr int kTailFlagWords = 1024;
bool tail_scratch(cudaStream_t stream, float** partials, uint32_t** counters);
// Zero the tail counters of the current device (after a device-side error, a
// launch may have left some set).
void reset_tail_flags();

// True when every pointer is an allocation of the current device (false for
// host, managed or another device's memory, and when that cannot be told).
bool operands_local(const void* const* ptrs, int n);
// Whether gemm_bf16 runs multicast clusters for these operands: asked for by
// the flag, or chosen for short K without pairs -- and only over memory of the
// current device.
bool bf16_uses_multicast(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                         bool pair, bool mcast_flag);

// Tail split (K pieces per leftover tile, 1 = none) the dense bf16 kernel
// uses for this shape on the context's device; negative status on failure.
int bf16_tail_split(int64_t M, int64_t N, int64_t K, bool pair, DeviceCtx* ctx);

// Launchers (arguments already validated).  kind: kKindBf16 or a
// block-scaled kind (gemm_kinds.h).
int launch_gemm(int kind, const void* A, int64_t lda, const void* B, int64_t ldb,
                const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb, void* D,
                int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype, const Epi& epi,
                unsigned flags, cudaStream_t stream, DeviceCtx* ctx);

// Host checks of an epilogue description (no CUDA calls); fills `out`.
int check_epilogue(const tg_epilogue* epi, Epi* out);

int launch_gemm_bf16_impl(const void* A, int64_t lda, const void* B, int64_t ldb, void* D,
                          int64_t ldd, int M, int N, int K, int d_dtype, const Epi& epi,
                          bool pair, bool mcast, cudaStream_t stream, DeviceCtx* ctx);

// Re-pitch of dense bf16 operands (gemm_bf16.cu).  TMA boxes over rows that
// start only 16 bytes aligned straddle extra L2 lines and land ~40% slower;
// for products large enough to repay a copy, such operands are first copied
// into workspace rows of `kp` elements (128-byte pitch).
struct Bf16Repitch {
  bool a = false, b = false;
  int64_t kp = 0;
  size_t bytes = 0;  // workspace bytes; 0: no re-pitch
};
// pair_clusters: the launch runs multicast clusters of two CTA pairs, which
// take badly aligned rows as they are (no re-pitch).
Bf16Repitch bf16_repitch_plan(int64_t lda, int64_t ldb, int64_t M, int64_t N, int64_t K,
                              bool pair_clusters);
int launch_gemm_bf16_repitched(const Bf16Repitch& rp, const void* A, int64_t lda, const void* B,
                               int64_t ldb, void* D, int64_t ldd, int M, int N, int K,
                               int d_dtype, const Epi& epi, bool pair, bool mcast,
                               void* workspace, cudaStream_t stream, DeviceCtx* ctx);

// no_scratch: the caller must not allocate (the static-scratch entry point),
// so nothing that allocates (the tail split's scratch) may be turned on.
int launch_gemm_mxfp8_impl(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int M, int N, int K, int d_dtype,
                           const Epi& epi, bool pair, bool mcast, uint8_t* sf_workspace,
                           cudaStream_t stream, DeviceCtx* ctx, bool no_scratch = false);

// Any block-scaled kind; sf_workspace holds blockscaled_workspace_bytes().
int launch_gemm_blockscaled_impl(int kind, const void* A, int64_t lda, const void* B,
                                 int64_t ldb, const void* SFA, int64_t ld_sfa, const void* SFB,
                                 int64_t ld_sfb, void* D, int64_t ldd, int M, int N, int K,
                                 int d_dtype, const Epi& epi, bool pair, bool mcast,
                                 uint8_t* sf_workspace, cudaStream_t stream, DeviceCtx* ctx,
                                 bool no_scratch = false);

// Host-side argument checks of a block-scaled call of `kind` (no CUDA calls).
int check_blockscaled_args(int kind, const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           int epilogue, unsigned flags);
inline int check_mxfp8_args(const void* A, int64_t lda, const void* B, int64_t ldb,
                            const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                            void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                            int epilogue, unsigned flags) {
  return check_blockscaled_args(kKindMxf8, A, lda, B, ldb, SFA, ld_sfa, SFB, ld_sfb, D, ldd, M,
                                N, K, d_dtype, epilogue, flags);
}

// Bytes of scale-image workspace a block-scaled problem needs (CTA pairs and
// multicast clusters share one image layout).
size_t blockscaled_workspace_bytes(int kind, int64_t M, int64_t N, int64_t K, bool pair);
size_t mxfp8_workspace_bytes(int64_t M, int64_t N, int64_t K, bool pair);

// bf16 GEMM with A rows gathered by row_idx (device int32 [M]).
int launch_gemm_bf16_gather_impl(const void* A, int64_t lda, int a_rows, const int* row_idx,
                                 int M, const void* B, int64_t ldb, void* D, int64_t ldd, int N,
                                 int K, int d_dtype, const Epi& epi, bool pair,
                                 cudaStream_t stream, DeviceCtx* ctx);

// Same product through a gathered copy of the rows in `workspace`
// (gather_workspace_bytes) and the dense kernel.
int launch_gemm_bf16_pregather_impl(const void* A, int64_t lda, int a_rows, const int* row_idx,
                                    int M, const void* B, int64_t ldb, void* D, int64_t ldd,
                                    int N, int K, int d_dtype, const Epi& epi, bool pair,
                                    void* workspace, cudaStream_t stream, DeviceCtx* ctx);
size_t gather_workspace_bytes(int64_t M, int64_t K);

// Skinny bf16 GEMM (M <= 128): split-K pieces reduce into an f32 target.
// `workspace` (f32, skinny_workspace_bytes) is used for bf16 D only.
int launch_gemm_skinny_impl(const void* A, int64_t lda, const void* B, int64_t ldb, void* D,
                            int64_t ldd, int M, int N, int K, int d_dtype, const Epi& epi,
                            int split_k, float* workspace, cudaStream_t stream, DeviceCtx* ctx);
size_t skinny_workspace_bytes(int64_t M, int64_t N, int d_dtype, int epi_op);
// K pieces per tile for split_k (0: automatic); *per_split = 64-element
// stages per piece.
int skinny_splits(int64_t N, int64_t K, int split_k, int num_sms, int* per_split);

// D = epilogue(0) when K == 0.
int launch_fill_epilogue(void* D, int64_t ldd, int64_t M, int64_t N, int d_dtype, const Epi& epi,
                         cudaStream_t stream);

int launch_transpose_b16(const void* in, int64_t ld_in, void* out, int64_t ld_out, int64_t rows,
                         int64_t cols, cudaStream_t stream, DeviceCtx* ctx);

}  // namespace tg
