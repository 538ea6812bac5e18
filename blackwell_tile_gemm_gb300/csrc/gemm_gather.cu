// bf16 GEMM with gathered A rows: D[i, :] = A[idx[i], :] * B^T (+ epilogue),
// the product of a mixture-of-experts layer, where the tokens routed to one
// expert are scattered over the activation matrix.
//
// The A tile is loaded with TMA tile::gather4 ("cp.async.bulk.tensor",
// section "Gather4 and scatter4": a 2-D map whose box is one row high, four
// runtime row coordinates per issue, a shared image of four box rows): the
// 32 lanes of the producer warp each gather four of the tile's 128 rows per
// stage into consecutive 128-byte rows of the stage buffer.  The 128-byte
// swizzle follows the shared address, so the buffer holds the same image a
// 128-row box load would, and the MMA, epilogue and B path are those of the
// dense kernel (single CTA or CTA pair).  Indices outside [0, rows of A)
// read a row past A's end, i.e. zeros.
//
// A gather4 occupies its issuing thread for tens of cycles, and the 32 per
// stage that a 128-row tile needs keep three issuing warps busier than the
// MMAs (8192^3-class shapes run at ~60% of the dense kernel).  The default
// path therefore gathers the rows into a workspace with a streaming copy
// first (2 * M * K * 2 bytes of extra traffic) and runs the dense kernel on
// it; TG_FLAG_GATHER_TMA selects the in-kernel gather4 path.
#include "gemm_launch.cuh"

namespace tg {

namespace {
using CfgGatherF32 = GemmCfg<1, kKindBf16, 256, 2, 4, false, false, true>;
using CfgGatherBf16 = GemmCfg<1, kKindBf16, 256, 2, 4, true, false, true>;
using CfgGatherPairF32 = GemmCfg<2, kKindBf16, 256, 2, 6, false, false, true>;
using CfgGatherPairBf16 = GemmCfg<2, kKindBf16, 256, 2, 6, true, false, true>;
// Row gather into a contiguous buffer: G[i, :] = A[idx[i], :] (zero rows for
// indices outside A).  One warp per row, 16-byte vectors (K % 8 == 0 and a
// 16-byte row stride, which the TMA row-stride rule already requires).
// One warp per gathered row: exactly K elements (16-byte vectors, then the
// last K % 8 one by one), so nothing past column K of A is read.
__global__ void gather_rows_kernel(const uint16_t* __restrict__ A, int64_t lda, int a_rows,
                                   const int* __restrict__ idx, int M, uint16_t* __restrict__ G,
                                   int64_t ldg, int K) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int kv = K / 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
       i < M; i += warps) {
    const int src = __ldg(idx + i);
    const bool valid = src >= 0 && src < a_rows;
    const uint16_t* a = A + static_cast<int64_t>(valid ? src : 0) * lda;
    uint16_t* g = G + i * ldg;
    const uint4* av = reinterpret_cast<const uint4*>(a);
    uint4* gv = reinterpret_cast<uint4*>(g);
    for (int k = lane; k < kv; k += 32) gv[k] = valid ? __ldg(av + k) : make_uint4(0u, 0u, 0u, 0u);
    const int t = kv * 8 + lane;
    if (lane < 8 && t < K) g[t] = valid ? a[t] : static_cast<uint16_t>(0);
  }
}

}  // namespace

// Gathered rows are written at a 128-byte pitch: TMA boxes over rows that
// are only 16-byte aligned land markedly slower.
size_t gather_workspace_bytes(int64_t M, int64_t K) {
  return static_cast<size_t>(M) * static_cast<size_t>((K + 63) / 64 * 64) * 2u;
}

int launch_gemm_bf16_pregather_impl(const void* A, int64_t lda, int a_rows, const int* row_idx,
                                    int M, const void* B, int64_t ldb, void* D, int64_t ldd,
                                    int N, int K, int d_dtype, const Epi& epi, bool pair,
                                    void* workspace, cudaStream_t stream, DeviceCtx* ctx) {
  const int64_t ldg = (K + 63) / 64 * 64;
  int64_t blocks = (static_cast<int64_t>(M) + 7) / 8;
  if (blocks > 16 * static_cast<int64_t>(ctx->num_sms)) blocks = 16 * ctx->num_sms;
  gather_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(A), lda, a_rows, row_idx, M,
      static_cast<uint16_t*>(workspace), ldg, K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  // The gathered rows live in this device's workspace; B decides whether the
  // short-K multicast clusters may run.
  const bool mcast = bf16_uses_multicast(workspace, B, M, N, K, pair, false);
  return launch_gemm_bf16_impl(workspace, ldg, B, ldb, D, ldd, M, N, K, d_dtype, epi, pair, mcast,
                               stream, ctx);
}

int launch_gemm_bf16_gather_impl(const void* A, int64_t lda, int a_rows, const int* row_idx,
                                 int M, const void* B, int64_t ldb, void* D, int64_t ldd, int N,
                                 int K, int d_dtype, const Epi& epi, bool pair,
                                 cudaStream_t stream, DeviceCtx* ctx) {
  constexpr int BN = 256;
  const int g = pair ? 2 : 1;
  CUtensorMap tA, tB;
  // Box one row high (the gather4 form); rows past a_rows read zeros.
  int rc = make_tensor_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, a_rows, lda * 2, 64, 1,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, ldb * 2, 64, BN / g,
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
  a.gather_idx = row_idx;
  a.gather_rows = a_rows;
  a.status = ctx->status;
  a.timeout_ns = wait_timeout_ns();
  const bool bf16_out = d_dtype == TG_D_BF16;
  if (!pair)
    return bf16_out ? launch_gemm_cfg<CfgGatherBf16>(tA, tB, tA, tB, a, stream, ctx)
                    : launch_gemm_cfg<CfgGatherF32>(tA, tB, tA, tB, a, stream, ctx);
  return bf16_out ? launch_gemm_cfg<CfgGatherPairBf16>(tA, tB, tA, tB, a, stream, ctx)
                  : launch_gemm_cfg<CfgGatherPairF32>(tA, tB, tA, tB, a, stream, ctx);
}

}  // namespace tg
