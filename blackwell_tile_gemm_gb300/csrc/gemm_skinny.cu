// Skinny bf16 GEMM: D[M,N] = A[M,K] * B[N,K]^T for M <= 128, the shape of a
// few activation rows against a large weight matrix.  Such a product is
// bound by reading B once from HBM (N*K*2 bytes), not by the tensor cores.
//
// The operands are swapped so that the large side fills the MMA's M: each
// work unit computes D^T[n0:n0+128, 0:Mp] = B[n0:n0+128, k-range] *
// A[0:Mp, k-range]^T with tcgen05.mma .kind::f16 M=128, N=Mp (Mp = M rounded
// up to 16, 32, 64 or 128; rows past M load as zeros).  N / 128 tiles alone
// would leave most SMs idle, so the K range of every tile is split into S
// pieces ("cp.async.bulk.tensor", section "Reductions": a tensor copy can add
// into global memory instead of overwriting it): each unit writes its f32
// partial tile to shared memory as [m][n] and reduces it into an f32 target
// [M, N] with one TMA reduce-add.  The target starts at the value of the
// epilogue's linear part (0, the constant, beta, or the column bias); a
// following pass applies SiLU and / or converts to bf16 when asked for.
// Partials arrive in a run-dependent order, so with S > 1 the last bits of D
// may differ between runs; S = 1 is deterministic.
//
// The three kernels of a call (initial value, GEMM, final pass) are chained
// with programmatic dependent launch, so the GEMM streams B while the
// initial value is written and the final pass is launched before the GEMM
// ends; each waits (griddepcontrol.wait) only where it reads what the
// previous kernel wrote.
//
// Roles (6 warps, one CTA per SM): warp 0 TMA producer, warp 1 TMEM
// allocator + MMA issuer, warps 2..5 epilogue (warp w reads TMEM lanes
// 32*(w%4).. = rows n of the tile).  Two accumulators of Mp columns let the
// next unit's MMAs run while the epilogue drains the last one.
#include "gemm_launch.cuh"

namespace tg {

namespace {

constexpr uint32_t kSiteSkEmpty = 21, kSiteSkFull = 22, kSiteSkAccEmpty = 23, kSiteSkAccFull = 24;

template <int kMp>
struct SkCfg {
  static constexpr int MP = kMp;                    // activation rows per tile (MMA N)
  static constexpr int W_BYTES = 128 * 128;         // 128 weight rows x 64 bf16
  static constexpr int X_BYTES = kMp * 128;         // Mp activation rows x 64 bf16
  static constexpr int STAGE_TX = W_BYTES + X_BYTES;
  static constexpr int OUT_BYTES = kMp * 128 * 4;   // f32 partial tile, [m][n]
  static constexpr int kFit = (200 * 1024 - OUT_BYTES) / STAGE_TX;
  static constexpr int kStages = kFit > 8 ? 8 : kFit;
  static constexpr int OFF_W = 0;
  static constexpr int OFF_X = OFF_W + kStages * W_BYTES;
  static constexpr int OFF_OUT = OFF_X + kStages * X_BYTES;
  static constexpr int OFF_BAR = OFF_OUT + OUT_BYTES;
  static constexpr int kAccBufs = 2;
  static constexpr int NUM_BARS = 2 * kStages + 2 * kAccBufs + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static constexpr int TMEM_COLS = 2 * kMp <= 32 ? 32 : 2 * kMp <= 64 ? 64 : 2 * kMp <= 128 ? 128 : 256;
  static constexpr int kEpiWarps = 4;
  static constexpr int kThreads = 64 + 32 * kEpiWarps;
  static_assert(kMp % 16 == 0 && kMp >= 16 && kMp <= 128, "MMA N");
  static_assert(kStages >= 3, "ring depth");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(OFF_X % 1024 == 0 && OFF_OUT % 1024 == 0, "swizzle atoms");
};

struct SkArgs {
  int num_n_tiles;
  int splits;        // K pieces per tile
  int per_split;     // stages (64 K each) per piece
  int stages_total;  // ceil(K / 64)
  float scale;       // factor on every partial (the AFFINE alpha; else 1)
  uint32_t* status;
  uint64_t timeout_ns;
};

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW,
                       const __grid_constant__ CUtensorMap tmX,
                       const __grid_constant__ CUtensorMap tmOut, const SkArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;                          // [kStages]  TMA -> MMA
  uint64_t* empty_bar = bars + C::kStages;            // [kStages]  MMA -> TMA
  uint64_t* accf_bar = bars + 2 * C::kStages;         // [2] MMA -> epilogue
  uint64_t* acce_bar = accf_bar + C::kAccBufs;        // [2] epilogue -> MMA
  uint64_t* drain_bar = acce_bar + C::kAccBufs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* epi_go = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  float* out = reinterpret_cast<float*>(smem + C::OFF_OUT);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], C::kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
    prefetch_tensormap(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, C::TMEM_COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  const WaitGuard guard{p.status, abort_flag, p.timeout_ns};
  const int num_units = p.num_n_tiles * p.splits;
  if (threadIdx.x == 0) griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();    // weights are read once
      const uint64_t pol_x = policy_evict_last();     // activations by every tile
      const uint32_t sW = smem_addr(smem + C::OFF_W);
      const uint32_t sX = smem_addr(smem + C::OFF_X);
      const uint32_t empty0 = smem_addr(&empty_bar[0]);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const int nt = u % p.num_n_tiles, sp = u / p.num_n_tiles;
        const int k0 = sp * p.per_split;
        const int k1 = min(k0 + p.per_split, p.stages_total);
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_try_wait(empty0 + 8u * stage, phase ^ 1u) &&
              !mbar_wait(&empty_bar[stage], phase ^ 1u, guard, kSiteSkEmpty)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_addr(&full_bar[stage]);
          mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_TX);
          tma_load_2d(sW + stage * C::W_BYTES, &tmW, fb, kb * 64, nt * 128, pol_w);
          tma_load_2d(sX + stage * C::X_BYTES, &tmX, fb, kb * 64, 0, pol_x);
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < C::kStages; ++s)
          if (issued & (1u << s))
            mbar_wait_drain(&full_bar[s], (issued_parity >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t wdesc0 =
          make_smem_desc(smem_addr(smem + C::OFF_W), 16, 1024, kDescSwizzle128B);
      const uint64_t xdesc0 =
          make_smem_desc(smem_addr(smem + C::OFF_X), 16, 1024, kDescSwizzle128B);
      const uint32_t full0 = smem_addr(&full_bar[0]);
      const uint32_t acce0 = smem_addr(&acce_bar[0]);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        const int sp = u / p.num_n_tiles;
        const int k0 = sp * p.per_split;
        const int k1 = min(k0 + p.per_split, p.stages_total);
        if (!mbar_try_wait(acce0 + 8u * acc, acc_phase ^ 1u) &&
            !mbar_wait(&acce_bar[acc], acc_phase ^ 1u, guard, kSiteSkAccEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::MP);
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_try_wait(full0 + 8u * stage, phase) &&
              !mbar_wait(&full_bar[stage], phase, guard, kSiteSkFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t wd = wdesc0 + static_cast<uint64_t>(stage * (C::W_BYTES >> 4));
          const uint64_t xd = xdesc0 + static_cast<uint64_t>(stage * (C::X_BYTES >> 4));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_bf16<1>(d_tmem, wd + 2 * k, xd + 2 * k, idesc_bf16_f32(128, C::MP),
                        (kb > k0 || k > 0) ? 1u : 0u);
          mma_commit(&empty_bar[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&accf_bar[acc]);
        if (++acc == C::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok || *abort_flag) {
        mma_commit(drain_bar);
        mbar_wait_drain(drain_bar, 0, p.timeout_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // One thread decides, for all four warps, whether a unit's accumulator
    // arrived, so that they all take the named barriers the same number of
    // times.
    const bool lead = warp == 2 && lane == 0;
    // Only the reduce into the target depends on the kernel that set its
    // initial value (launched just before, programmatically serialised).
    if (lead) griddep_wait();
    const uint32_t q = static_cast<uint32_t>(warp & 3);   // TMEM lanes 32q.. = tile rows
    const int n_local = static_cast<int>(32 * q + lane);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const int nt = u % p.num_n_tiles;
      if (lead) *epi_go = mbar_wait(&accf_bar[acc], acc_phase, guard, kSiteSkAccFull) ? 1 : 0;
      named_bar_sync(1, 32 * C::kEpiWarps);
      if (!*epi_go) break;
      tc_fence_after_sync();
      uint32_t v[C::MP];
      const uint32_t t_row = tmem_base + ((32u * q) << 16) + static_cast<uint32_t>(acc * C::MP);
#pragma unroll
      for (int c = 0; c < C::MP / 16; ++c) tmem_ld_32x32b_x16(t_row + 16 * c, v + 16 * c);
      tmem_ld_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_relaxed(&acce_bar[acc]);
      // The staging tile is free once the previous reduce has read it.
      if (lead) bulk_wait_group_read<0>();
      named_bar_sync(1, 32 * C::kEpiWarps);
#pragma unroll
      for (int m = 0; m < C::MP; ++m) out[m * 128 + n_local] = __uint_as_float(v[m]) * p.scale;
      fence_proxy_async_smem();
      named_bar_sync(1, 32 * C::kEpiWarps);
      if (lead) {
        tma_reduce_add_2d(&tmOut, smem_addr(out), nt * 128, 0);
        bulk_commit_group();
      }
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lead) bulk_wait_group0();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<1>(tmem_base, C::TMEM_COLS);
  }
}

// The f32 target starts at the linear part of the epilogue: T[m][n] = init.
__global__ void skinny_init_kernel(float* T, int64_t ldt, int M, int N, Epi epi) {
  griddep_launch_dependents();     // the GEMM may start streaming B meanwhile
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / N, n = i % N;
    float v = 0.0f;
    if (epi.op == kEpiAddScalar) v = epi.alpha;
    else if (epi.op == kEpiAffine) v = epi.beta;
    else if (epi_uses_bias(epi.op)) v = epi.bias[n];
    T[m * ldt + n] = v;
  }
}

// D[m][n] = post(T[m][n]): SiLU for the SiLU ops, then the conversion to D's
// type (T and D may be the same f32 array).
__global__ void skinny_finalize_kernel(const float* T, int64_t ldt, void* D, int64_t ldd, int M,
                                       int N, int bf16_out, Epi epi) {
  griddep_wait();                  // every partial of the GEMM has been added
  const int64_t total = static_cast<int64_t>(M) * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t m = i / N, n = i % N;
    float v = T[m * ldt + n];
    if (epi.op == kEpiSiluAffine) v = silu_f32(v) * epi.alpha + epi.beta;
    else if (epi.op == kEpiBiasColSilu) v = silu_f32(v);
    if (bf16_out)
      reinterpret_cast<uint16_t*>(D)[m * ldd + n] = static_cast<uint16_t>(pack_bf16x2(v, v) & 0xFFFFu);
    else
      reinterpret_cast<float*>(D)[m * ldd + n] = v;
  }
}

template <class C>
int launch_skinny_cfg(const CUtensorMap& tW, const CUtensorMap& tX, const CUtensorMap& tO,
                      const SkArgs& a, int units, cudaStream_t stream, DeviceCtx* ctx) {
  std::atomic<int>& slot = LaunchState<C>::units[ctx->device];
  if (slot.load(std::memory_order_acquire) == 0) {
    cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return cuda_fail(e);
    slot.store(1, std::memory_order_release);
  }
  const int grid = units < ctx->num_sms ? units : ctx->num_sms;
  cudaLaunchConfig_t cfg{};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<C>, tW, tX, tO, a);
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

int elementwise_grid(int64_t total, DeviceCtx* ctx) {
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = 8 * static_cast<int64_t>(ctx->num_sms);
  return static_cast<int>(blocks < 1 ? 1 : blocks > cap ? cap : blocks);
}

}  // namespace

int skinny_splits(int64_t N, int64_t K, int split_k, int num_sms, int* per_split) {
  const int n_tiles = ceil_div_i(N, 128);
  const int total = ceil_div_i(K, 64);
  int s = split_k;
  if (s <= 0) {
    // Units (tile, piece) run in waves of num_sms; the time is about
    // waves * stages-per-piece, the work n_tiles * total stages, so
    // fill = work / (num_sms * waves * per).  Pieces keep at least 4 stages
    // (each unit ends with an epilogue and a partial-tile reduce) and at
    // most 32 per tile; the smallest count within 1% of the best fill wins.
    double fill[33] = {};
    double best = 0.0;
    for (int c = 1; c <= 32 && c <= total; ++c) {
      const int per = (total + c - 1) / c;
      if (c > 1 && per < 4) break;
      const int pieces = (total + per - 1) / per;
      const int64_t units = static_cast<int64_t>(n_tiles) * pieces;
      const int64_t waves = (units + num_sms - 1) / num_sms;
      fill[c] = static_cast<double>(n_tiles) * total /
                (static_cast<double>(num_sms) * static_cast<double>(waves) * per);
      if (fill[c] > best) best = fill[c];
    }
    s = 1;
    for (int c = 1; c <= 32; ++c)
      if (fill[c] >= best - 0.01) {
        s = c;
        break;
      }
  }
  if (s < 1) s = 1;
  if (s > total) s = total;
  const int per = (total + s - 1) / s;
  *per_split = per;
  return (total + per - 1) / per;   // no empty pieces
}

// f32 D is its own reduction target when its rows end on a 16-byte boundary
// (N % 4 == 0).  A reduce whose box crosses a ragged column N may touch the
// caller's row padding up to the next 16-byte boundary, so ragged f32 D and
// bf16 D go through an f32 workspace of 16-byte rows and a finalize pass.
bool skinny_direct(int64_t N, int d_dtype) { return d_dtype == TG_D_F32 && N % 4 == 0; }

size_t skinny_workspace_bytes(int64_t M, int64_t N, int d_dtype, int epi_op) {
  const bool direct = skinny_direct(N, d_dtype);
  (void)epi_op;
  return direct ? 0 : static_cast<size_t>(M) * static_cast<size_t>((N + 3) / 4 * 4) * 4u;
}

int launch_gemm_skinny_impl(const void* A, int64_t lda, const void* B, int64_t ldb, void* D,
                            int64_t ldd, int M, int N, int K, int d_dtype, const Epi& epi,
                            int split_k, float* workspace, cudaStream_t stream, DeviceCtx* ctx) {
  const int mp = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
  SkArgs a{};
  a.num_n_tiles = ceil_div_i(N, 128);
  a.stages_total = ceil_div_i(K, 64);
  a.splits = skinny_splits(N, K, split_k, ctx->num_sms, &a.per_split);
  a.scale = epi.op == kEpiAffine ? epi.alpha : 1.0f;
  a.status = ctx->status;
  a.timeout_ns = wait_timeout_ns();
  const bool direct = skinny_direct(N, d_dtype);
  float* T = direct ? static_cast<float*>(D) : workspace;
  const int64_t ldt = direct ? ldd : (N + 3) / 4 * 4;
  const int64_t total = static_cast<int64_t>(M) * N;
  skinny_init_kernel<<<elementwise_grid(total, ctx), 256, 0, stream>>>(T, ldt, M, N, epi);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);

  CUtensorMap tW, tX, tO;
  int rc = make_tensor_map_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, K, N, ldb * 2, 64, 128,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, M, lda * 2, 64, mp,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != TG_OK) return rc;
  rc = make_tensor_map_2d(&tO, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, T, N, M, ldt * 4, 128, mp,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc != TG_OK) return rc;
  const int units = a.num_n_tiles * a.splits;
  switch (mp) {
    case 16: rc = launch_skinny_cfg<SkCfg<16>>(tW, tX, tO, a, units, stream, ctx); break;
    case 32: rc = launch_skinny_cfg<SkCfg<32>>(tW, tX, tO, a, units, stream, ctx); break;
    case 64: rc = launch_skinny_cfg<SkCfg<64>>(tW, tX, tO, a, units, stream, ctx); break;
    default: rc = launch_skinny_cfg<SkCfg<128>>(tW, tX, tO, a, units, stream, ctx); break;
  }
  if (rc != TG_OK) return rc;
  const bool post = !direct || epi.op == kEpiSiluAffine || epi.op == kEpiBiasColSilu;
  if (post) {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(elementwise_grid(total, ctx)), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const float* Tc = T;
    const int bf16_out = d_dtype == TG_D_BF16 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, skinny_finalize_kernel, Tc, ldt, D, ldd, M, N, bf16_out, epi);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return TG_OK;
}

}  // namespace tg
