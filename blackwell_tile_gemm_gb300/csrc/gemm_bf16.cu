// Dense bf16 GEMM configurations (kind::f16, f32 accumulation).
//
//   single CTA : 128 x 256 tiles, 4-stage ring of 48 KB, two 256-column
//                accumulators in tensor memory (all 512 columns).
//   CTA pair   : 256 x 256 tiles per cluster of two (cta_group::2), each CTA
//                stages 128 rows of A and 128 rows of B per stage (32 KB),
//                6-stage ring, two accumulators per CTA.
//   multicast  : clusters of two CTA pairs on vertically adjacent tiles; each
//                CTA loads a 64-row quarter of the shared B tile and
//                multicasts it to its counterpart in the other pair.
#include "gemm_launch.cuh"

namespace tg {

namespace {
using CfgF32 = GemmCfg<1, kKindBf16, 256, 2, 4, false>;
using CfgBf16 = GemmCfg<1, kKindBf16, 256, 2, 4, true>;
using CfgPairF32 = GemmCfg<2, kKindBf16, 256, 2, 6, false>;
using CfgPairBf16 = GemmCfg<2, kKindBf16, 256, 2, 6, true>;
// Clusters of two CTA pairs multicasting the shared B tile (TG_FLAG_MULTICAST).
using CfgPairMcF32 = GemmCfg<2, kKindBf16, 256, 2, 6, false, true>;
using CfgPairMcBf16 = GemmCfg<2, kKindBf16, 256, 2, 6, true, true>;
// Clusters of two single CTAs on vertically adjacent tiles multicasting the
// shared B tile (each loads 128 of its 256 rows).
using CfgMcF32 = GemmCfg<1, kKindBf16, 256, 2, 4, false, true>;
using CfgMcBf16 = GemmCfg<1, kKindBf16, 256, 2, 4, true, true>;
}  // namespace

bool single_cta_multicast_pays(int64_t M, int64_t N, int64_t K) {
  return K <= 1536 && M >= 3000 && N >= 3000;
}

// Multicast clusters, asked for (TG_FLAG_MULTICAST) or chosen for short K,
// load the shared B tile with .multicast::cluster TMA.  They run only when A
// and B are allocations of the current device, so that a multicast tensor map
// never covers another GPU's (or the host's) memory; otherwise the plain
// pair or single-CTA kernel computes the same result.
bool bf16_uses_multicast(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                         bool pair, bool mcast_flag) {
  if (!mcast_flag && (pair || !single_cta_multicast_pays(M, N, K))) return false;
  const void* ops[2] = {A, B};
  return operands_local(ops, 2);
}

int launch_gemm_bf16_impl(const void* A, int64_t lda, const void* B, int64_t ldb, void* D,
                          int64_t ldd, int M, int N, int K, int d_dtype, const Epi& epi,
                          bool pair, bool mcast, cudaStream_t stream, DeviceCtx* ctx) {
  constexpr int BN = 256;
  const int g = pair ? 2 : 1;
  const int b_rows = BN / g;
  CUtensorMap tA, tB;
  int rc = make_tensor_map_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, 64, 128,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  const int b_box = mcast ? b_rows / 2 : b_rows;
  rc = make_tensor_map_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, ldb * 2, 64, b_box,
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
  a.status = ctx->status;
  a.timeout_ns = wait_timeout_ns();
  const bool bf16_out = d_dtype == TG_D_BF16;
  // Single CTAs: for short K on large products, clusters of two sharing the
  // B tile by multicast cut each CTA's loads from 48 to 32 KB a stage
  // (graph replay: 4096^2 x 512 23.9 -> 18.4 us, 4096^2 x 1024 32.6 ->
  // 27.8, 8192^2 x 1024 96.6 -> 90.5, 4000 x 3000 x 1000 28.6 -> 27.0); at
  // K >= 2048 the coupled rings cost more than they save (4096^3 89 -> 95).
  if (!pair && mcast)
    return bf16_out ? launch_gemm_cfg<CfgMcBf16>(tA, tB, tA, tB, a, stream, ctx)
                    : launch_gemm_cfg<CfgMcF32>(tA, tB, tA, tB, a, stream, ctx);
  if (!pair)
    return bf16_out ? launch_gemm_cfg<CfgBf16>(tA, tB, tA, tB, a, stream, ctx)
                    : launch_gemm_cfg<CfgF32>(tA, tB, tA, tB, a, stream, ctx);
  if (mcast)
    return bf16_out ? launch_gemm_cfg<CfgPairMcBf16>(tA, tB, tA, tB, a, stream, ctx)
                    : launch_gemm_cfg<CfgPairMcF32>(tA, tB, tA, tB, a, stream, ctx);
  return bf16_out ? launch_gemm_cfg<CfgPairBf16>(tA, tB, tA, tB, a, stream, ctx)
                  : launch_gemm_cfg<CfgPairF32>(tA, tB, tA, tB, a, stream, ctx);
}

int bf16_tail_split(int64_t M, int64_t N, int64_t K, bool pair, DeviceCtx* ctx) {
  // Clusters never split (operands in this device's memory pick them for
  // short K).
  if (!pair && single_cta_multicast_pays(M, N, K)) return 1;
  const int g = pair ? 2 : 1;
  const int num_tiles = ceil_div_i(M, 128 * g) * ceil_div_i(N, 256);
  const int units_max =
      pair ? gemm_units_for_device<CfgPairF32>(ctx) : gemm_units_for_device<CfgF32>(ctx);
  if (units_max < 0) return -TG_ERR_CUDA;
  int W = 0, R = 0;
  return pair ? tail_split_for<CfgPairF32>(num_tiles, ceil_div_i(K, 64), units_max, &W, &R)
              : tail_split_for<CfgF32>(num_tiles, ceil_div_i(K, 64), units_max, &W, &R);
}

// ---------------------------------------------------------------------------
// Re-pitch.  Measured on GB300 (4000 x 3000 x 1000, graph replay): rows of
// 2000 bytes (16-byte aligned) 37.5 us, 2016 (32-byte) 30.6 us, 1984
// (64-byte) 27.1 us, 2048 (128-byte) 26.8 us: a 128-byte box row that
// straddles L2 lines lands late.  Copying A (and B) to rows of a 128-byte
// pitch costs ~4 bytes per element of HBM or L2 traffic; for 16-byte rows
// it pays when the product is large against its operands, M*N/(M+N) >=
// 1250.  For 32-byte rows the copy cost more than it saved (8192^2 x 1000,
// 2016-byte rows: 108 -> 118 us).  Multicast clusters of two CTA pairs load
// half as many B boxes, and there the copy no longer pays (graph replay,
// 16-byte rows, with -> without the copy: 4000 x 3000 x 1000 26.8 -> 24.4
// us, 6000^2 x 3000 136 -> 125 us, 8192^2 x 8000 at 8008-element rows 645
// -> ~615 us; 8192^2 x 1000 107.1 -> 108.8 us), while plain pairs and
// single CTAs still gain 10-15% from it at those shapes.

namespace {

// Rows [0, a_rows) come from A, the next b_rows from B, one warp per row:
// exactly K elements (16-byte vectors, four per lane in flight, then the
// last K % 8 one by one), so that nothing past column K is read.
__global__ void repitch_rows_kernel(const uint16_t* __restrict__ a, int64_t lda, int a_rows,
                                    const uint16_t* __restrict__ b, int64_t ldb, int b_rows,
                                    uint16_t* __restrict__ dst, int64_t ld_dst, int K) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t total = static_cast<int64_t>(a_rows) + b_rows;
  const int kv = K / 8;
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5);
       r < total; r += warps) {
    const bool from_a = r < a_rows;
    const uint16_t* s = from_a ? a + r * lda : b + (r - a_rows) * ldb;
    uint16_t* d = dst + r * ld_dst;
    const uint4* sv = reinterpret_cast<const uint4*>(s);
    uint4* dv = reinterpret_cast<uint4*>(d);
    for (int k0 = 0; k0 < kv; k0 += 128) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + 32 * u + lane;
        if (k < kv) v[u] = __ldcs(sv + k);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = k0 + 32 * u + lane;
        if (k < kv) dv[k] = v[u];
      }
    }
    const int t = kv * 8 + lane;
    if (lane < 8 && t < K) d[t] = s[t];
  }
}

// 0: rows 64-byte aligned (or better); else the alignment class in bytes.
int row_alignment_class(int64_t ld) {
  const int64_t b = ld * 2;
  return b % 64 == 0 ? 0 : b % 32 == 0 ? 32 : 16;
}

}  // namespace

Bf16Repitch bf16_repitch_plan(int64_t lda, int64_t ldb, int64_t M, int64_t N, int64_t K,
                              bool pair_clusters) {
  Bf16Repitch rp;
  if (pair_clusters || K < 128 || M <= 0 || N <= 0) return rp;
  const double ratio = static_cast<double>(M) * static_cast<double>(N) / static_cast<double>(M + N);
  auto wants = [&](int64_t ld) { return row_alignment_class(ld) == 16 && ratio >= 1250.0; };
  rp.a = wants(lda);
  rp.b = wants(ldb);
  if (!rp.a && !rp.b) return rp;
  rp.kp = (K + 63) / 64 * 64;
  rp.bytes = static_cast<size_t>((rp.a ? M : 0) + (rp.b ? N : 0)) * static_cast<size_t>(rp.kp) * 2u;
  return rp;
}

int launch_gemm_bf16_repitched(const Bf16Repitch& rp, const void* A, int64_t lda, const void* B,
                               int64_t ldb, void* D, int64_t ldd, int M, int N, int K,
                               int d_dtype, const Epi& epi, bool pair, bool mcast,
                               void* workspace, cudaStream_t stream, DeviceCtx* ctx) {
  // Workspace: A's rows (if re-pitched), then B's, each kp elements.
  uint16_t* w = static_cast<uint16_t*>(workspace);
  const int a_rows = rp.a ? M : 0, b_rows = rp.b ? N : 0;
  int64_t blocks = (static_cast<int64_t>(a_rows) + b_rows + 7) / 8;
  if (blocks > 16 * static_cast<int64_t>(ctx->num_sms)) blocks = 16 * ctx->num_sms;
  repitch_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint16_t*>(A), lda, a_rows, static_cast<const uint16_t*>(B), ldb, b_rows,
      w, rp.kp, K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  if (rp.a) {
    A = w;
    lda = rp.kp;
  }
  if (rp.b) {
    B = w + static_cast<int64_t>(a_rows) * rp.kp;
    ldb = rp.kp;
  }
  return launch_gemm_bf16_impl(A, lda, B, ldb, D, ldd, M, N, K, d_dtype, epi, pair, mcast,
                               stream, ctx);
}

// ---------------------------------------------------------------------------
// K == 0: D = epilogue(0)
// ---------------------------------------------------------------------------

namespace {
__global__ void fill_kernel(void* D, int64_t ldd, int64_t M, int64_t N, int bf16_out, Epi epi) {
  const int64_t total = M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / N, c = i % N;
    float y = 0.0f;
    if (epi.op == kEpiAddScalar)
      y = epi.alpha;
    else if (epi.op != kEpiNone)
      y = apply_epi_general(epi.op, epi.alpha, epi.beta, 0.0f,
                            epi_uses_bias(epi.op) ? epi.bias[c] : 0.0f);
    if (bf16_out)
      reinterpret_cast<uint16_t*>(D)[r * ldd + c] =
          static_cast<uint16_t>(pack_bf16x2(y, y) & 0xFFFFu);
    else
      reinterpret_cast<float*>(D)[r * ldd + c] = y;
  }
}
}  // namespace

int launch_fill_epilogue(void* D, int64_t ldd, int64_t M, int64_t N, int d_dtype, const Epi& epi,
                         cudaStream_t stream) {
  const int64_t total = M * N;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(D, ldd, M, N,
                                                                 d_dtype == TG_D_BF16, epi);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

}  // namespace tg
