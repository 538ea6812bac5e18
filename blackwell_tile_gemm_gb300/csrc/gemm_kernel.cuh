// Persistent, warp-specialised tcgen05 GEMM: D[M,N] = A[M,K] * B[N,K]^T.
//
// The operation and its operand roles follow "tcgen05.mma" (TVM TIRx tile
// operation guide), sections "Operands and repeat axes" (per-CTA canonical
// shapes D (M/g, N), A (M/g, K), B (N/g, K); SFB carries the full N in each
// CTA of a pair), "Shared descriptors are byte-stride contracts" (K-major,
// 128-byte swizzled rows, next 8-row group at SDO) and "Examples" (explicit K
// decomposition into K16 issues, one commit per issue sequence, tcgen05.ld
// 32x32b read-back).  TMA staging follows "cp.async.bulk.tensor" (one elected
// thread, mbarrier with expected transaction bytes, out-of-range boxes read
// zeros).  The pages leave pipelining, election and scheduling to the caller;
// this file is that caller code:
//
//   warp 0      TMA producer: one lane waits for a free ring slot, posts the
//               expected bytes and issues the A / B (and scale-image) loads.
//   warp 1      TMEM allocator and MMA issuer: one lane waits for a full slot
//               (block-scaled: for its scales in TMEM), issues the four MMAs
//               of 32 bytes of K each, and commits to the slot's "empty"
//               barrier; at the end of a tile it commits to the accumulator's
//               "full" barrier.
//   warps 2..9  epilogue: wait for a full accumulator; each warp owns 32
//               TMEM lanes (rows) x BN/2 columns.  With two accumulators it
//               reads one 32-row x 128-byte box at a time (tcgen05.ld,
//               row = lane), applies the fused op, converts, stages the box
//               128B-swizzled in shared memory and stores it with a TMA tile
//               store, handing the accumulator back after its last read.
//               With one accumulator (block-scaled kinds) it reads its whole
//               share at once and hands the accumulator back, then stores
//               each chunk through 32-row x 64-byte staged boxes with TMA
//               (where shared memory allows; else, and for chunks that cross
//               column N, from registers with st.global.v4).
//   warps 10,11 block-scaled kinds only: scale copiers; once a stage's data
//               has landed, each copies half of its scale images into the
//               stage's TMEM scale columns (tcgen05.cp) and commits to the
//               stage's "scales ready" barrier, which the MMAs wait for.
//
// Tiles are visited persistently (one MMA unit -- a CTA, or a CTA pair --
// per SM or SM pair, static stride) in grouped order so that units running at
// the same time share A and B panels in L2; multicast clusters pair two units
// on vertically adjacent tiles that share the B tile; the last wave's tiles
// may be cut into K pieces (tail split, see next_work).  Every wait is
// bounded (see tg_ptx.cuh: mbar_wait).
#pragma once

#include <cstdint>
#include <cuda.h>

#include "epilogue.cuh"
#include "tg_ptx.cuh"

namespace tg {

enum : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaFull = 2,
  kSiteMmaAccEmpty = 3,
  kSiteEpiAccFull = 4,
  kSiteScaleFull = 5,
};

struct GemmArgs {
  int M, N, K;
  int num_m_tiles;  // tiles of kCtaGroup*128 rows
  int num_n_tiles;  // tiles of BN columns
  int num_k_blocks; // stages of BK elements
  void* D;
  int64_t ldd;
  Epi epi;          // fused elementwise epilogue
  int sfa_blocks;   // 128-row blocks per K group in the SFA image
  int sfb_blocks;   // 128-row blocks per K group in the SFB image
  int raster_group; // m-tiles per band of the tile order
  // Tile order refinements (see tile_coords and next_work): n_snake walks the
  // n-tiles of every other band backwards, so that consecutive bands start on
  // the B panels the previous one ended on; k_snake walks K backwards in every
  // other wave of whole tiles, so that a unit's next tile starts on the K
  // slices the units around it read last (a plain LRU-like cache holds those,
  // and evicts the first slices just before the next wave would reuse them).
  int n_snake;
  int k_snake;
  const int* gather_idx;  // gathered A: D row i uses A row gather_idx[i] (else null)
  int gather_rows;        // rows of A; indices outside [0, gather_rows) read zeros
  // Tail split (see next_work): tiles below full_tiles are whole work items;
  // with tail_split = S > 1 the tail_items = R * S items that follow are K
  // pieces of the R last tiles.  Every epilogue warp of every piece writes
  // its share of the piece's f32 partial tile to partials and then arrives on
  // its share's counter; the arrival that completes the count (the S-th)
  // adds the S partials in piece order, stores D and sets the counter back
  // to 0, so that every launch (also a graph replay) starts from zeroed
  // counters.  No piece waits for another.
  int full_tiles;
  int tail_split;
  int tail_items;
  float* partials;        // [tail tile][piece][CTA of pair][BN cols][128 rows] f32
  uint32_t* counters;     // [tail tile][CTA of pair][epilogue warp], 0 between launches
  uint32_t* status;
  uint64_t timeout_ns;
  // Host side only (the kernel ignores it): the call must not allocate, so
  // the launcher never turns on the tail split, whose scratch is allocated.
  bool no_scratch;
  // SM clock readout: when set, the MMA thread of each unit adds its SM
  // cycles, nanoseconds and 1 to these three sums (tg_kernel_clock_record).
  unsigned long long* clk;
};

// kKind_: kKindBf16 (dense bf16) or one of the block-scaled kinds kKindMxf8,
// kKindMxf4, kKindNvf4 (tg_ptx.cuh).
template <int kCtaGroup_, int kKind_, int kBN_, int kAccBufs_, int kStages_, bool kBf16Out_,
          bool kMcast_ = false, bool kGather_ = false>
struct GemmCfg {
  // Gathered A: the producer warp loads the A tile row by row with
  // tile::gather4 (32 lanes x 4 rows = 128 rows), from GemmArgs::gather_idx.
  static constexpr bool kGather = kGather_;
  static constexpr int kCtaGroup = kCtaGroup_;
  // Multicast: clusters of two CTA pairs that work on vertically adjacent
  // tiles share the B tile; each CTA loads a quarter of it and multicasts
  // the quarter to its counterpart in the other pair.
  static constexpr bool kMcast = kMcast_;
  static constexpr int kPairs = kMcast ? 2 : 1;           // MMA units per cluster
  static constexpr int kClusterCtas = kCtaGroup * kPairs;
  static constexpr int kKind = kKind_;
  static constexpr bool kMx = kKind != kKindBf16;   // block-scaled
  // Scale layout per stage (128 bytes of K per row = 4 MMAs of 32 bytes):
  // an MMA reads kSfVec scales per row, so a stage needs kSfVec 512-byte
  // images of 128 rows x 4 scale bytes per 128-row block.
  static constexpr int kSfVec = scale_vec_of(kKind);
  static constexpr int kSfGroups = kSfVec;
  static constexpr int BM = 128;                    // D rows per CTA (TMEM lanes)
  static constexpr int BN = kBN_;                   // D columns per tile (MMA N)
  static constexpr int kAccBufs = kAccBufs_;
  static constexpr int kStages = kStages_;
  static constexpr bool kBf16Out = kBf16Out_;
  // Tensor-map elements per stage along K (128 bytes: 64 bf16 or 128 one-byte
  // elements; a packed-FP4 map is addressed in bytes, 2 values each).
  static constexpr int BK = kMx ? 128 : 64;
  static constexpr int kIssues = 4;                 // MMAs of 32 bytes of K per stage
  static constexpr int B_ROWS = BN / kCtaGroup;     // B rows this CTA stages
  static constexpr int B_LOAD_ROWS = B_ROWS / kPairs;  // B rows this CTA loads
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = B_ROWS * 128;
  static constexpr int kSfBlocksB = BN / 128;       // 128-row blocks of SFB per tile
  static constexpr int SFA_BYTES = kSfGroups * 512;
  static constexpr int SFB_BYTES = kSfGroups * kSfBlocksB * 512;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // shared memory carve-up (offsets from a 1024-aligned base)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + kStages * A_BYTES;
  static constexpr int OFF_SFA = OFF_B + kStages * B_BYTES;
  static constexpr int OFF_SFB = OFF_SFA + kStages * SFA_BYTES;
  // Block-scaled kinds: two warps copy the scales into TMEM, each issuing
  // half of a stage's tcgen05.cp.  A copy costs its issuing thread ~80
  // cycles before the next one issues, while copies from different warps
  // proceed in parallel, and none of them delays MMAs issued by another warp;
  // so the copies leave the MMA thread, and two issuers keep up with the 12
  // copies an NVFP4 stage needs within the 512 cycles of its MMAs.
  static constexpr int kSfWarps = kMx ? 2 : 0;
  static constexpr int NUM_BARS =
      (kMx ? 3 : 2) * kStages + 2 * kAccBufs + 1 + kSfWarps;
  // TMA-store epilogue, where shared memory allows: each epilogue warp
  // stages one box of 32 rows at a time and one lane stores it with TMA.
  // With two accumulators the boxes are 128 bytes wide (32 f32 or 64 bf16
  // columns, 128B swizzle) and are read from TMEM box by box; the
  // block-scaled rings (one accumulator, which their epilogue must hand back
  // as early as possible) read everything first and stage 64-byte boxes
  // (64B swizzle), whose 2 KB per warp fit beside the MXFP8 ring.  Without
  // room (the MXFP4 pair ring) the warps store from registers with
  // st.global.v4.
  static constexpr int OFF_SF_END = OFF_SFB + kStages * SFB_BYTES;
  // Staged box rows: 128 bytes with two accumulators (box-wise epilogue),
  // 64 bytes with one (the whole share is read first; 2 KB per warp fits
  // beside the block-scaled rings).
  static constexpr int kStgRowBytes = kAccBufs == 2 ? 128 : 64;
  static constexpr int kStgWarpBytes = 32 * kStgRowBytes;
  static constexpr int OFF_STG = (OFF_SF_END + 1023) & ~1023;
  static constexpr bool kTmaStore =
      OFF_STG + 8 * kStgWarpBytes + NUM_BARS * 8 + 16 + 1024 <= 227 * 1024;
  static constexpr int OFF_BAR = kTmaStore ? OFF_STG + 8 * kStgWarpBytes : ((OFF_SF_END + 7) & ~7);
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  // tensor memory columns
  static constexpr int ACC_COLS = BN;
  static constexpr int SFA_COLS = 4 * kSfGroups;
  static constexpr int SFB_COLS = 4 * kSfGroups * kSfBlocksB;
  static constexpr int SF_COL0 = ACC_COLS * kAccBufs;
  static constexpr int SF_STAGE_COLS = SFA_COLS + SFB_COLS;
  static constexpr int TMEM_USED = SF_COL0 + SF_STAGE_COLS * kStages;
  static constexpr int TMEM_COLS = TMEM_USED <= 32    ? 32
                                   : TMEM_USED <= 64  ? 64
                                   : TMEM_USED <= 128 ? 128
                                   : TMEM_USED <= 256 ? 256
                                                      : 512;
  static constexpr uint32_t MMA_M = BM * kCtaGroup;
  // Epilogue: 8 warps; warp w reads TMEM lanes 32*(w%4).. and one half of the
  // BN columns, holding that half (BN/2 f32 per thread) in registers.
  static constexpr int kEpiWarps = 8;
  static constexpr int kEpiCols = BN / 2;
  static constexpr int kEpiChunks = kEpiCols / 32;
  static constexpr int kSfWarp0 = 2 + kEpiWarps;    // first scale-copy warp
  // Gathered A: warps 0 and kGatherWarp0.. issue the tile's 32 gather4 loads
  // per stage together (a gather4 occupies its issuing thread for tens of
  // cycles, so one warp cannot keep up with the MMAs).
  static constexpr int kGatherWarps = kGather ? 3 : 1;
  static constexpr int kGatherWarp0 = kSfWarp0 + kSfWarps;
  static constexpr int kThreads = 64 + 32 * kEpiWarps + 32 * kSfWarps + 32 * (kGatherWarps - 1);
  static_assert(TMEM_USED <= 512, "tensor memory has 512 columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "MMA N");
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms");
  static_assert(!kMcast || kCtaGroup == 2 || !kMx, "single-CTA multicast clusters: bf16 only");
  static_assert(!kMx || BN % 128 == 0, "scale images cover 128-row blocks of B");
  static_assert(!kGather || (!kMx && !kMcast), "gathered A: bf16, without multicast");
};

// One work item of a unit: a whole tile, or one K piece of a tail tile.
struct Work {
  int t;        // tile id (tile order)
  int k0;       // first K stage
  int ks;       // step between K stages (negative: backwards)
  int nk;       // number of K stages: k0, k0 + ks, ..., k0 + (nk - 1) * ks
  int piece;    // K piece (its partial's slot; the order in which partials add up)
  int tail;     // tail tile index, or -1 for a whole tile
};

// Item i of `unit`: tiles unit, unit + U, ... below full_tiles; then, with a
// tail split, the unit's one K piece of a tail tile.  Every unit runs full
// waves of whole tiles (full_tiles = W * U), and the R tiles a last, partial
// wave would leave to R units are cut into S pieces run by R * S units.  The
// pieces never wait for each other: the last one to finish adds the partial
// tiles and stores D, so the result does not depend on which units of the
// grid are resident at the same time.
__device__ __forceinline__ bool next_work(const GemmArgs& p, int unit, int num_units, int i,
                                          Work& w) {
  const int t = unit + i * num_units;
  if (t < p.full_tiles) {
    w.t = t;
    const bool back = p.k_snake && (i & 1);
    w.k0 = back ? p.num_k_blocks - 1 : 0;
    w.ks = back ? -1 : 1;
    w.nk = p.num_k_blocks;
    w.piece = 0;
    w.tail = -1;
    return true;
  }
  if (p.tail_split <= 1 || i != p.full_tiles / num_units || unit >= p.tail_items) return false;
  // Piece q takes stages q, q + S, q + 2S, ...: the S pieces of a tile then
  // read neighbouring 128-byte chunks of each row at any moment.  (Pieces of
  // contiguous K ranges kept fixed 2-4 KB offsets between them and ran 2-4x
  // slower per SM, their loads landing on the same L2 slices.)
  const int S = p.tail_split;
  w.tail = unit / S;
  w.piece = unit % S;
  w.t = p.full_tiles + w.tail;
  w.k0 = w.piece;
  w.ks = S;
  w.nk = (p.num_k_blocks - w.piece + S - 1) / S;
  return true;
}

// Grouped tile order: consecutive tile ids walk down a band of `group`
// m-tiles before moving to the next n-tile, so the CTAs that run at the same
// time share a few A and B panels in L2.
__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group, int n_snake,
                                            int& tm, int& tn) {
  const int per_group = group * num_n;
  const int g = t / per_group;
  const int first_m = g * group;
  const int gm = min(num_m - first_m, group);
  const int r = t - g * per_group;
  tm = first_m + r % gm;
  tn = r / gm;
  if (n_snake && (g & 1)) tn = num_n - 1 - tn;
}

// Copies one stage's scale images from shared memory into its TMEM scale
// columns (32 rows x 16 bytes per copy, replicated into the four 32-lane
// slabs; 8-row groups 128 bytes apart).  Shared layout per stage: SFA
// [group][512 B], SFB [block][group][512 B].  TMEM layout from column sfa_t:
// SFA group g at 4g; SFB group g, block b at SFA_COLS + 4 (g * blocks + b),
// so that the blocks of one group are adjacent columns, as an MMA of N = BN
// reads them (row r of SFB in byte column 4 (r / 32) + sf).
// The copies are numbered SFA images first, then SFB (block, image); copier
// `part` of kSfWarps issues those whose number is part modulo kSfWarps.
template <class C>
__device__ __forceinline__ void copy_stage_scales(uint32_t sfa_t, uint64_t sfadesc0,
                                                  uint64_t sfbdesc0, int stage, int part) {
#pragma unroll
  for (int g = 0; g < C::kSfGroups; ++g)
    if (g % C::kSfWarps == part)
      tmem_cp_32x128b_warpx4<C::kCtaGroup>(
          sfa_t + 4 * g, sfadesc0 + static_cast<uint64_t>((stage * C::SFA_BYTES + 512 * g) >> 4));
#pragma unroll
  for (int b = 0; b < C::kSfBlocksB; ++b)
#pragma unroll
    for (int g = 0; g < C::kSfGroups; ++g)
      if ((C::kSfGroups + b * C::kSfGroups + g) % C::kSfWarps == part)
        tmem_cp_32x128b_warpx4<C::kCtaGroup>(
            sfa_t + C::SFA_COLS + 4 * (g * C::kSfBlocksB + b),
            sfbdesc0 + static_cast<uint64_t>(
                           (stage * C::SFB_BYTES + 512 * (b * C::kSfGroups + g)) >> 4));
}

// Four column biases starting at `c` (zeros past N).
__device__ __forceinline__ float4 bias4(const GemmArgs& p, int c) {
  if (c + 4 <= p.N) {
    const uint4 q = ld_global_nc_v4(p.epi.bias + c);   // same address in every lane
    return make_float4(__uint_as_float(q.x), __uint_as_float(q.y), __uint_as_float(q.z),
                       __uint_as_float(q.w));
  }
  float t[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) t[e] = c + e < p.N ? p.epi.bias[c + e] : 0.0f;
  return make_float4(t[0], t[1], t[2], t[3]);
}

// SILU_AFFINE / AFFINE / BIAS_COL / BIAS_COL_SILU on 32 accumulator columns
// [col0, col0+32) of one row, in place.  The op is uniform over the launch,
// so each branch below runs without divergence.
__device__ __forceinline__ void epilogue_general_chunk(const GemmArgs& p, int col0,
                                                       uint32_t (&v)[32]) {
  const int op = p.epi.op;
  const float alpha = p.epi.alpha, beta = p.epi.beta;
  if (op == kEpiAffine) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = __float_as_uint(apply_epi_general(kEpiAffine, alpha, beta,
                                               __uint_as_float(v[i]), 0.0f));
    return;
  }
  if (op == kEpiSiluAffine) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      v[i] = __float_as_uint(apply_epi_general(kEpiSiluAffine, alpha, beta,
                                               __uint_as_float(v[i]), 0.0f));
    return;
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 b = bias4(p, col0 + 4 * q);
    const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      v[4 * q + e] = __float_as_uint(
          apply_epi_general(op, alpha, beta, __uint_as_float(v[4 * q + e]), bb[e]));
  }
}

// Stores 32 columns [col0, col0+32) of one row as D = v (+ add when kAdd),
// 4 (f32) or 8 (bf16) columns per 16-byte store.
template <class C, bool kAdd>
__device__ __forceinline__ void epilogue_store_chunk(const GemmArgs& p, int row, int col0,
                                                     const uint32_t (&v)[32], float add,
                                                     uint64_t pol) {
  if constexpr (C::kBf16Out) {
    uint16_t* drow = reinterpret_cast<uint16_t*>(p.D) + static_cast<int64_t>(row) * p.ldd;
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = kAdd ? pack_bf16x2(__uint_as_float(v[2 * i]) + add,
                                __uint_as_float(v[2 * i + 1]) + add)
                  : pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    if (col0 + 32 <= p.N) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_global_v4_hint(drow + col0 + 8 * i, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3],
                          pol);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = col0 + 8 * i;
        if (c + 8 <= p.N) {
          st_global_v4_hint(drow + c, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3], pol);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (c + e < p.N)
              drow[c + e] = static_cast<uint16_t>(w[4 * i + e / 2] >> (16 * (e & 1)));
        }
      }
    }
  } else {
    float* drow = reinterpret_cast<float*>(p.D) + static_cast<int64_t>(row) * p.ldd;
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = kAdd ? __float_as_uint(__uint_as_float(v[i]) + add) : v[i];
    if (col0 + 32 <= p.N) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        st_global_v4_hint(drow + col0 + 4 * i, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3],
                          pol);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = col0 + 4 * i;
        if (c + 4 <= p.N) {
          st_global_v4_hint(drow + c, w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3], pol);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (c + e < p.N) drow[c + e] = __uint_as_float(w[4 * i + e]);
        }
      }
    }
  }
}

// TMA-store epilogue: writes one 32-row x 128-byte box of D (lane = row)
// into this warp's staging buffer, 128B-swizzled: 16-byte piece j of row r
// sits at r*128 + ((j ^ (r & 7)) * 16), so the eight lanes of each quarter
// warp write eight different bank groups.  The box holds 32 f32 columns
// (chunk va) or 64 bf16 columns (chunks va, vb).  stg_row = buffer + lane*128.
template <class C, bool kAdd>
__device__ __forceinline__ void epilogue_stage_box(uint32_t stg_row, uint32_t lane,
                                                   const uint32_t (&va)[32],
                                                   const uint32_t (&vb)[32], float add) {
  const uint32_t sw = lane & 7u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
    if constexpr (C::kBf16Out) {
      const uint32_t(&src)[32] = j < 4 ? va : vb;
      const int c0 = 8 * (j & 3);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = __uint_as_float(src[c0 + 2 * e]);
        const float x1 = __uint_as_float(src[c0 + 2 * e + 1]);
        w[e] = kAdd ? pack_bf16x2(x0 + add, x1 + add) : pack_bf16x2(x0, x1);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = kAdd ? __float_as_uint(__uint_as_float(va[4 * j + e]) + add) : va[4 * j + e];
    }
    st_shared_v4(stg_row + ((static_cast<uint32_t>(j) ^ sw) << 4), w[0], w[1], w[2], w[3]);
  }
}

// One 32-row x 64-byte box (lane = row) of chunk v into the warp's staging
// buffer, 64B-swizzled: 16-byte piece j of row r at r*64 + ((j ^ ((r >> 1) &
// 3)) * 16).  bf16: the chunk's 32 columns; f32: columns 16h .. 16h+15.
template <class C>
__device__ __forceinline__ void epilogue_stage_box64(uint32_t stg_row, uint32_t lane,
                                                     const uint32_t (&v)[32], int h, float add) {
  const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w[4];
    if constexpr (C::kBf16Out) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_bf16x2(__uint_as_float(v[8 * j + 2 * e]) + add,
                           __uint_as_float(v[8 * j + 2 * e + 1]) + add);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = __float_as_uint(__uint_as_float(v[16 * h + 4 * j + e]) + add);
    }
    st_shared_v4(stg_row + ((static_cast<uint32_t>(j) ^ sw) << 4), w[0], w[1], w[2], w[3]);
  }
}

template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSFA,
                        const __grid_constant__ CUtensorMap tmSFB,
                        const __grid_constant__ CUtensorMap tmD, const GemmArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full_bar = bars;                          // [kStages]  TMA -> MMA
  uint64_t* empty_bar = bars + C::kStages;            // [kStages]  MMA -> TMA
  uint64_t* accf_bar = bars + 2 * C::kStages;         // [kAccBufs] MMA -> epilogue
  uint64_t* acce_bar = accf_bar + C::kAccBufs;        // [kAccBufs] epilogue -> MMA
  uint64_t* drain_bar = acce_bar + C::kAccBufs;       // MMA completion on give-up
  uint64_t* sfr_bar = drain_bar + 1;                  // [kStages] scales in TMEM -> MMA
  uint64_t* sf_drain_bar = sfr_bar + C::kStages;      // [kSfWarps] copies on give-up
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = threadIdx.x & 31;
  // An MMA unit is a CTA pair (cta_group::2) or a single CTA; a multicast
  // cluster holds two units on vertically adjacent tiles.
  const uint32_t rank = (C::kClusterCtas > 1) ? cluster_ctarank() : 0u;
  const uint32_t pair_rank = C::kCtaGroup == 2 ? (rank & 1u) : 0u;  // 0: MMA-issuing CTA
  const uint32_t pair_id = rank / C::kCtaGroup;       // which unit of the cluster
  const uint32_t lead_rank = rank - pair_rank;        // rank of this unit's leader
  const bool leader = pair_rank == 0;
  // tcgen05.commit multicast masks: this unit, and every CTA whose loads
  // land in this unit's shared memory (the whole cluster under multicast).
  const uint16_t pair_mask =
      static_cast<uint16_t>((C::kCtaGroup == 2 ? 3u : 1u) << lead_rank);
  const uint16_t stage_mask =
      C::kMcast ? static_cast<uint16_t>((1u << C::kClusterCtas) - 1u) : pair_mask;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], C::kPairs);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&accf_bar[b], 1);
      mbar_init(&acce_bar[b], C::kEpiWarps * C::kCtaGroup);
    }
    mbar_init(drain_bar, 1);
    if constexpr (C::kMx) {
      for (int s = 0; s < C::kStages; ++s) mbar_init(&sfr_bar[s], C::kSfWarps);
      for (int w = 0; w < C::kSfWarps; ++w) mbar_init(&sf_drain_bar[w], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if constexpr (C::kMx) {
      prefetch_tensormap(&tmSFA);
      prefetch_tensormap(&tmSFB);
    }
    if constexpr (C::kTmaStore) prefetch_tensormap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc<C::kCtaGroup>(tmem_slot, C::TMEM_COLS);
    tmem_relinquish<C::kCtaGroup>();
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::kClusterCtas > 1) cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // Programmatic dependent launch: everything above is on-chip, so it may
  // overlap the end of the kernel before this one in the stream; operands,
  // D and the scratch are touched only once that kernel has completed and
  // its writes are visible.
  griddep_wait();

  const WaitGuard guard{p.status, abort_flag, p.timeout_ns};
  // Work units: tiles of kPairs x 256 rows (one per cluster) by BN columns.
  const int num_mc = (p.num_m_tiles + C::kPairs - 1) / C::kPairs;
  const int unit = blockIdx.x / C::kClusterCtas;      // cluster index
  const int num_units = gridDim.x / C::kClusterCtas;

  // The producer and MMA loops run one thread each and are latency-critical:
  // the tensor pipe queues only a couple of MMAs, so every instruction the
  // MMA thread spends between issues can idle it.  Hence barrier checks take
  // an inline fast path (one try_wait) and fall back to the bounded wait only
  // when a barrier is not ready, shared-memory descriptors are advanced by
  // adding offsets, and the next stage's barrier is probed while the current
  // stage's MMAs are queued.
  if (C::kGather && (warp == 0 || (warp >= C::kGatherWarp0 &&
                                    warp < C::kGatherWarp0 + C::kGatherWarps - 1))) {
    // ------------------------------------------------ producer, gathered A
    // kGatherWarps warps (gw = 0 .. kGatherWarps-1): each waits for a free
    // slot itself; warp 0 posts the expected bytes and loads the B tile.
    // Gather op j (rows 4j .. 4j+3 of the A tile, j < 32) belongs to warp
    // j % kGatherWarps, lane j / kGatherWarps, which keeps the op's four row
    // indices in registers for the tile.
    if constexpr (C::kGather) {
      const int gw = warp == 0 ? 0 : warp - C::kGatherWarp0 + 1;
      const int op = gw + C::kGatherWarps * static_cast<int>(lane);
      const bool has_op = op < 32;
      const uint64_t pol_ab = policy_evict_last();
      const uint32_t sA = smem_addr(smem + C::OFF_A);
      const uint32_t sB = smem_addr(smem + C::OFF_B);
      const uint32_t empty0 = smem_addr(&empty_bar[0]);
      const uint32_t full0 = smem_addr(&full_bar[0]);
      const uint32_t full_dst0 = C::kCtaGroup == 2 ? map_to_cta(full0, lead_rank) : full0;
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;
      bool ok = true;
      Work w;
      for (int it = 0; ok && next_work(p, unit, num_units, it, w); ++it) {
        const int t = w.t;
        int tmc, tn;
        tile_coords(t, num_mc, p.num_n_tiles, p.raster_group, p.n_snake, tmc, tn);
        const int tm = tmc * C::kPairs + static_cast<int>(pair_id);
        const int a_row = tm * C::MMA_M + static_cast<int>(pair_rank) * C::BM;
        const int b_row = tn * C::BN + static_cast<int>(pair_rank) * C::B_ROWS;
        int r[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = a_row + 4 * op + j;
          int src = has_op && i < p.M ? p.gather_idx[i] : p.gather_rows;
          // Any index outside A is sent past its end, where the load reads zeros.
          if (src < 0 || src >= p.gather_rows) src = p.gather_rows;
          r[j] = src;
        }
        for (int j = 0, kb = w.k0; j < w.nk; ++j, kb += w.ks) {
          int got = 1;
          if (lane == 0)
            got = (mbar_try_wait(empty0 + 8u * stage, phase ^ 1u) ||
                   mbar_wait(&empty_bar[stage], phase ^ 1u, guard, kSiteProducerEmpty))
                      ? 1
                      : 0;
          got = __shfl_sync(0xFFFFFFFFu, got, 0);
          if (!got) {
            ok = false;
            break;
          }
          const int kx = kb * C::BK;
          const uint32_t fb = full_dst0 + 8u * stage;
          if (gw == 0 && lane == 0) {
            if constexpr (C::kCtaGroup == 1) {
              mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_TX);
            } else {
              if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * C::STAGE_TX);
            }
          }
          __syncwarp();
          const uint32_t dstA = sA + stage * C::A_BYTES + static_cast<uint32_t>(op) * 512u;
          if constexpr (C::kCtaGroup == 1) {
            if (has_op) tma_gather4_2d(dstA, &tmA, fb, kx, r[0], r[1], r[2], r[3], pol_ab);
            if (gw == 0 && lane == 0)
              tma_load_2d(sB + stage * C::B_BYTES, &tmB, fb, kx, b_row, pol_ab);
          } else {
            if (has_op) tma_gather4_2d_pair(dstA, &tmA, fb, kx, r[0], r[1], r[2], r[3], pol_ab);
            if (gw == 0 && lane == 0)
              tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, fb, kx, b_row, pol_ab);
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load of this CTA is issued: the next kernel in the stream may
      // start its prologue on SMs this grid frees.
      if (warp == 0 && lane == 0) griddep_launch_dependents();
      if (!ok && leader && lane == 0) {
        for (int s = 0; s < C::kStages; ++s)
          if (issued & (1u << s))
            mbar_wait_drain(&full_bar[s], (issued_parity >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_ab = policy_evict_last();
      const uint32_t sA = smem_addr(smem + C::OFF_A);
      const uint32_t sB = smem_addr(smem + C::OFF_B);
      const uint32_t sSFA = smem_addr(smem + C::OFF_SFA);
      const uint32_t sSFB = smem_addr(smem + C::OFF_SFB);
      const uint32_t empty0 = smem_addr(&empty_bar[0]);
      const uint32_t full0 = smem_addr(&full_bar[0]);
      // Pair: both CTAs' loads complete on the leader's barrier.
      const uint32_t full_dst0 = C::kCtaGroup == 2 ? map_to_cta(full0, lead_rank) : full0;
      // The same CTA of the other unit: rank ^ kCtaGroup.
      const uint16_t mcast_mask = static_cast<uint16_t>(
          (1u << rank) | (1u << (rank ^ static_cast<uint32_t>(C::kCtaGroup))));
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;   // per-stage bit masks
      bool ok = true;
      Work w;
      for (int it = 0; ok && next_work(p, unit, num_units, it, w); ++it) {
        const int t = w.t;
        int tmc, tn;
        tile_coords(t, num_mc, p.num_n_tiles, p.raster_group, p.n_snake, tmc, tn);
        const int tm = tmc * C::kPairs + static_cast<int>(pair_id);
        const int a_row = tm * C::MMA_M + static_cast<int>(pair_rank) * C::BM;
        const int b_row = tn * C::BN + static_cast<int>(pair_rank) * C::B_ROWS;
        const int sfa_row = C::kCtaGroup == 2 ? tm * 2 + static_cast<int>(pair_rank) : tm;
        const int sfb_row = tn * (C::BN / 128);
        for (int j = 0, kb = w.k0; j < w.nk; ++j, kb += w.ks) {
          if (!mbar_try_wait(empty0 + 8u * stage, phase ^ 1u) &&
              !mbar_wait(&empty_bar[stage], phase ^ 1u, guard, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const int kx = kb * C::BK;
          const uint32_t fb = full_dst0 + 8u * stage;
          if constexpr (C::kCtaGroup == 1) {
            mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_TX);
            tma_load_2d(sA + stage * C::A_BYTES, &tmA, fb, kx, a_row, pol_ab);
            if constexpr (C::kMcast) {
              // This CTA's half of the B tile, into itself and the other
              // CTA of the cluster (same offset in both).
              tma_load_2d_mcast(sB + stage * C::B_BYTES + pair_id * (C::B_LOAD_ROWS * 128), &tmB,
                                fb, kx, b_row + static_cast<int>(pair_id) * C::B_LOAD_ROWS,
                                mcast_mask, pol_ab);
            } else {
              tma_load_2d(sB + stage * C::B_BYTES, &tmB, fb, kx, b_row, pol_ab);
            }
            if constexpr (C::kMx) {
              tma_load_2d(sSFA + stage * C::SFA_BYTES, &tmSFA, fb, 0, kb * p.sfa_blocks + sfa_row,
                          pol_ab);
              tma_load_2d(sSFB + stage * C::SFB_BYTES, &tmSFB, fb, 0, kb * p.sfb_blocks + sfb_row,
                          pol_ab);
            }
          } else {
            // Only the leader posts the expected byte count (for the pair).
            if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * C::STAGE_TX);
            tma_load_2d_pair(sA + stage * C::A_BYTES, &tmA, fb, kx, a_row, pol_ab);
            if constexpr (C::kMcast) {
              // This CTA's quarter of the B tile, into itself and its
              // counterpart in the other pair (same offset in both).
              tma_load_2d_pair_mcast(
                  sB + stage * C::B_BYTES + pair_id * (C::B_LOAD_ROWS * 128), &tmB, fb, kx,
                  b_row + static_cast<int>(pair_id) * C::B_LOAD_ROWS, mcast_mask, pol_ab);
            } else {
              tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, fb, kx, b_row, pol_ab);
            }
            if constexpr (C::kMx) {
              tma_load_2d_pair(sSFA + stage * C::SFA_BYTES, &tmSFA, fb, 0,
                               kb * p.sfa_blocks + sfa_row, pol_ab);
              tma_load_2d_pair(sSFB + stage * C::SFB_BYTES, &tmSFB, fb, 0,
                               kb * p.sfb_blocks + sfb_row, pol_ab);
            }
          }
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load of this CTA is issued: the next kernel in the stream may
      // start its prologue on SMs this grid frees.
      griddep_launch_dependents();
      if (!ok && leader) {
        // Gave up: let the loads already issued land before the CTA exits.
        for (int s = 0; s < C::kStages; ++s)
          if (issued & (1u << s))
            mbar_wait_drain(&full_bar[s], (issued_parity >> s) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      const unsigned long long clk_c0 = clock64();
      const uint64_t clk_g0 = global_timer_ns();
      const uint32_t acce0 = smem_addr(&acce_bar[0]);
      // K-major, 128-byte swizzled operands: 8-row groups 1024 bytes apart;
      // MMA k of a stage reads the 32-byte K slice k of each row.
      const uint64_t adesc0 =
          make_smem_desc(smem_addr(smem + C::OFF_A), 16, 1024, kDescSwizzle128B);
      const uint64_t bdesc0 =
          make_smem_desc(smem_addr(smem + C::OFF_B), 16, 1024, kDescSwizzle128B);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool ready = false;       // ready barrier of `stage` already seen complete
      // The MMAs of a stage wait for its TMA data, or with a scale warp for
      // its scales in TMEM (which that warp copies after the data landed).
      uint64_t* ready_bar = C::kMx ? sfr_bar : full_bar;
      const uint32_t ready0 = smem_addr(&ready_bar[0]);
      Work w;
      for (int it = 0; ok && next_work(p, unit, num_units, it, w); ++it) {
        if (!mbar_try_wait(acce0 + 8u * acc, acc_phase ^ 1u) &&
            !mbar_wait(&acce_bar[acc], acc_phase ^ 1u, guard, kSiteMmaAccEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::ACC_COLS);
        for (int j = 0, kb = w.k0; j < w.nk; ++j, kb += w.ks) {
          if (!ready && !mbar_try_wait(ready0 + 8u * stage, phase) &&
              !mbar_wait(&ready_bar[stage], phase, guard, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const int ns = stage + 1 == C::kStages ? 0 : stage + 1;
          const uint32_t nph = stage + 1 == C::kStages ? phase ^ 1u : phase;
          const uint64_t ad = adesc0 + static_cast<uint64_t>(stage * (C::A_BYTES >> 4));
          const uint64_t bd = bdesc0 + static_cast<uint64_t>(stage * (C::B_BYTES >> 4));
          if constexpr (C::kMx) {
            const uint32_t sfa_t = tmem_base + C::SF_COL0 + stage * C::SF_STAGE_COLS;
            const uint32_t sfb_t = sfa_t + C::SFA_COLS;
#pragma unroll
            for (int k = 0; k < C::kIssues; ++k) {
              // MMA k reads kSfVec scales per row starting at scale k * kSfVec
              // of the stage: image g, byte offset (scale-factor id) sf.
              const int g = (k * C::kSfVec) / 4, sf = (k * C::kSfVec) % 4;
              mma_block_scaled<C::kCtaGroup, C::kKind>(
                  d_tmem, ad + 2 * k, bd + 2 * k,
                  idesc_block_scaled<C::kKind>(C::MMA_M, C::BN, sf, sf), sfa_t + 4 * g,
                  sfb_t + 4 * g * C::kSfBlocksB, (j != 0 || k != 0));
              if (k == 0) ready = mbar_try_wait(ready0 + 8u * ns, nph);
            }
          } else {
#pragma unroll
            for (int k = 0; k < C::kIssues; ++k) {
              mma_bf16<C::kCtaGroup>(d_tmem, ad + 2 * k, bd + 2 * k,
                                     idesc_bf16_f32(C::MMA_M, C::BN), (j != 0 || k != 0));
              if (k == 0) ready = mbar_try_wait(ready0 + 8u * ns, nph);
            }
          }
          if constexpr (C::kCtaGroup == 1 && C::kMcast)
            mma_commit_mc(&empty_bar[stage], stage_mask);
          else if constexpr (C::kCtaGroup == 1)
            mma_commit(&empty_bar[stage]);
          else
            mma_commit_pair(&empty_bar[stage], stage_mask);
          stage = ns;
          phase = nph;
        }
        if (!ok) break;
        if constexpr (C::kCtaGroup == 1)
          mma_commit(&accf_bar[acc]);
        else
          mma_commit_pair(&accf_bar[acc], pair_mask);
        if (++acc == C::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (p.clk != nullptr) {
        atomicAdd(p.clk, static_cast<unsigned long long>(clock64()) - clk_c0);
        atomicAdd(p.clk + 1, static_cast<unsigned long long>(global_timer_ns() - clk_g0));
        atomicAdd(p.clk + 2, 1ull);
      }
      if (!ok || *abort_flag) {
        // Gave up: wait until every MMA issued so far has finished with
        // shared and tensor memory before they are released.
        if constexpr (C::kCtaGroup == 1)
          mma_commit(drain_bar);
        else
          mma_commit_pair(drain_bar, static_cast<uint16_t>(1u << lead_rank));
        mbar_wait_drain(drain_bar, 0, p.timeout_ns);
      }
    }
  } else if (C::kMx && warp >= C::kSfWarp0 && warp < C::kSfWarp0 + C::kSfWarps) {
    // ------------------------------------------------------------ scale copiers
    if constexpr (C::kMx) {
      const int part = warp - C::kSfWarp0;
      if (lane == 0 && leader) {
        const uint64_t sfadesc0 =
            make_smem_desc(smem_addr(smem + C::OFF_SFA), 16, 128, kDescSwizzleNone);
        const uint64_t sfbdesc0 =
            make_smem_desc(smem_addr(smem + C::OFF_SFB), 16, 128, kDescSwizzleNone);
        const uint32_t full0 = smem_addr(&full_bar[0]);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        bool copied = false;
        Work w;
        for (int it = 0; ok && next_work(p, unit, num_units, it, w); ++it) {
          for (int j = 0, kb = w.k0; j < w.nk; ++j, kb += w.ks) {
            if (!mbar_try_wait(full0 + 8u * stage, phase) &&
                !mbar_wait(&full_bar[stage], phase, guard, kSiteScaleFull)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            copy_stage_scales<C>(tmem_base + C::SF_COL0 + stage * C::SF_STAGE_COLS, sfadesc0,
                                 sfbdesc0, stage, part);
            if constexpr (C::kCtaGroup == 1)
              mma_commit(&sfr_bar[stage]);
            else
              mma_commit_pair(&sfr_bar[stage], static_cast<uint16_t>(1u << lead_rank));
            copied = true;
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (copied && (!ok || *abort_flag)) {
          // Gave up: the copies already issued finish before TMEM is freed.
          if constexpr (C::kCtaGroup == 1)
            mma_commit(&sf_drain_bar[part]);
          else
            mma_commit_pair(&sf_drain_bar[part], static_cast<uint16_t>(1u << lead_rank));
          mbar_wait_drain(&sf_drain_bar[part], 0, p.timeout_ns);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int slab = warp & 3;                        // TMEM lanes 32*slab .. +31
    const int half = (warp - 2) >> 2;                 // which BN/2 columns
    const int row_in_tile = slab * 32 + static_cast<int>(lane);
    const uint64_t pol_d = policy_evict_first();      // D is written once: keep A/B in L2
    // NONE and ADD_SCALAR are folded into the stores; the other ops first
    // transform the registers in place.
    const bool epi_lean = p.epi.op == kEpiNone || p.epi.op == kEpiAddScalar;
    const float epi_add = p.epi.op == kEpiAddScalar ? p.epi.alpha : 0.0f;
    // This warp's staging buffer for the TMA-store epilogue.
    const uint32_t stg =
        smem_addr(smem + C::OFF_STG) + static_cast<uint32_t>(warp - 2) * C::kStgWarpBytes;
    const uint32_t stg_row = stg + lane * static_cast<uint32_t>(C::kStgRowBytes);
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t acce_remote = 0;
    if constexpr (C::kCtaGroup == 2) acce_remote = map_to_cta(smem_addr(&acce_bar[0]), lead_rank);
    Work w;
    for (int it = 0; next_work(p, unit, num_units, it, w); ++it) {
      int tmc, tn;
      tile_coords(w.t, num_mc, p.num_n_tiles, p.raster_group, p.n_snake, tmc, tn);
      const int tm = tmc * C::kPairs + static_cast<int>(pair_id);
      // One lane waits for the accumulator; the others wait at the warp barrier.
      int got = 1;
      if (lane == 0) got = mbar_wait(&accf_bar[acc], acc_phase, guard, kSiteEpiAccFull) ? 1 : 0;
      got = __shfl_sync(0xFFFFFFFFu, got, 0);
      if (!got) break;
      tc_fence_after_sync();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(slab * 32) << 16) +
                             static_cast<uint32_t>(acc * C::ACC_COLS + half * C::kEpiCols);
      if constexpr (C::kTmaStore && C::kAccBufs == 2) {
        // Box-wise: the accumulator is read one box (32 rows x 128 bytes of
        // D) at a time, which keeps 32 or 64 values live instead of 128; the
        // second accumulator buffer lets the MMA warp run ahead meanwhile.
        // The buffer goes back after its last read.
        constexpr int kPerBox = C::kBf16Out ? 2 : 1;   // accumulator chunks per box
        constexpr int kBoxes = C::kEpiChunks / kPerBox;
        const int row0 = tm * C::MMA_M + static_cast<int>(pair_rank) * C::BM + slab * 32;
        const int col_base = tn * C::BN + half * C::kEpiCols;
        // Tail split.  A partial tile is stored column-major, [BN][128] f32:
        // the 32 lanes of a warp (32 consecutive rows) then write and read 128
        // contiguous bytes per column.  part_col(q) points at this thread's
        // row in the first of its columns in piece q's partial.
        const int S = p.tail_split;
        auto part_col = [&](int piece) {
          return p.partials +
                 ((static_cast<int64_t>(w.tail) * S + piece) * C::kCtaGroup + pair_rank) *
                     (128 * C::BN) +
                 static_cast<int64_t>(half * C::kEpiCols) * 128 + row_in_tile;
        };
        bool store_d = true;
        if (w.tail >= 0) {
          // Publish this piece's share of the partial tile, then arrive on
          // the share's counter (one per epilogue warp of each CTA).
          float* dst = part_col(w.piece);
#pragma unroll
          for (int b = 0; b < kBoxes; ++b) {
            uint32_t vb[kPerBox][32];
#pragma unroll
            for (int h = 0; h < kPerBox; ++h)
              tmem_ld_32x32b_x32(t_row + 32 * (kPerBox * b + h), vb[h]);
            tmem_ld_wait();
            if (b == kBoxes - 1) {
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) {
                if constexpr (C::kCtaGroup == 1)
                  mbar_arrive_relaxed(&acce_bar[acc]);
                else
                  mbar_arrive_relaxed_cluster(acce_remote + 8u * static_cast<uint32_t>(acc));
              }
            }
#pragma unroll
            for (int h = 0; h < kPerBox; ++h)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                __stcg(dst + (32 * (kPerBox * b + h) + i) * 128, __uint_as_float(vb[h][i]));
          }
          // Every lane's partial stores are ordered before lane 0's arrival.
          __threadfence();
          __syncwarp();
          uint32_t* counter =
              p.counters + (static_cast<int64_t>(w.tail) * C::kCtaGroup + pair_rank) * C::kEpiWarps +
              (warp - 2);
          uint32_t prev = 0;
          if (lane == 0) prev = arrive_counter_gpu(counter);
          prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
          store_d = prev == static_cast<uint32_t>(S - 1);
          if (store_d) {
            // The last arrival: every other piece's share is published.
            // Nobody touches the counter again in this launch.
            __threadfence();
            if (lane == 0) *counter = 0u;
          }
        }
        if (store_d) {
#pragma unroll
          for (int b = 0; b < kBoxes; ++b) {
            uint32_t vb[kPerBox][32];
            if (w.tail < 0) {
#pragma unroll
              for (int h = 0; h < kPerBox; ++h)
                tmem_ld_32x32b_x32(t_row + 32 * (kPerBox * b + h), vb[h]);
              tmem_ld_wait();
              if (b == kBoxes - 1) {
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                  if constexpr (C::kCtaGroup == 1)
                    mbar_arrive_relaxed(&acce_bar[acc]);
                  else
                    mbar_arrive_relaxed_cluster(acce_remote + 8u * static_cast<uint32_t>(acc));
                }
              }
            } else {
              // The pieces' partials, added in piece order 0, 1, ..., S-1
              // whichever piece arrived last, so repeated calls give the
              // same bits.
              const float* src0 = part_col(0);
#pragma unroll
              for (int h = 0; h < kPerBox; ++h)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  vb[h][i] = __float_as_uint(__ldcg(src0 + (32 * (kPerBox * b + h) + i) * 128));
              for (int q = 1; q < S; ++q) {
                const float* src = part_col(q);
#pragma unroll
                for (int h = 0; h < kPerBox; ++h)
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    vb[h][i] = __float_as_uint(__uint_as_float(vb[h][i]) +
                                               __ldcg(src + (32 * (kPerBox * b + h) + i) * 128));
              }
            }
            const int col0 = col_base + 32 * kPerBox * b;
            if (row0 < p.M && col0 < p.N) {
              if (!epi_lean) {
#pragma unroll
                for (int h = 0; h < kPerBox; ++h)
                  if (col0 + 32 * h < p.N) epilogue_general_chunk(p, col0 + 32 * h, vb[h]);
              }
              if (col0 + 32 * kPerBox <= p.N) {
                // The previous box's store has finished reading the buffer.
                if (lane == 0) bulk_wait_group_read0();
                __syncwarp();
                if (epi_lean)
                  epilogue_stage_box<C, true>(stg_row, lane, vb[0], vb[kPerBox - 1], epi_add);
                else
                  epilogue_stage_box<C, false>(stg_row, lane, vb[0], vb[kPerBox - 1], 0.0f);
                fence_proxy_async_smem();
                __syncwarp();
                // Rows >= M are clipped by the store.
                if (lane == 0) {
                  tma_store_2d_hint(&tmD, stg, col0, row0, pol_d);
                  bulk_commit_group();
                }
              } else {
                // The box crosses column N: a clipped TMA store may write up to
                // the next 16-byte boundary past N, into the caller's row
                // padding, so the ragged box is stored from registers.
                const int row = row0 + static_cast<int>(lane);
#pragma unroll
                for (int h = 0; h < kPerBox; ++h)
                  if (row < p.M && col0 + 32 * h < p.N) {
                    if (epi_lean)
                      epilogue_store_chunk<C, true>(p, row, col0 + 32 * h, vb[h], epi_add, pol_d);
                    else
                      epilogue_store_chunk<C, false>(p, row, col0 + 32 * h, vb[h], 0.0f, pol_d);
                  }
              }
            }
          }
        }
      } else {
        // Read this warp's whole share of the accumulator, then hand the
        // accumulator back to the MMA warp before converting and storing.
        uint32_t v[C::kEpiChunks][32];
#pragma unroll
        for (int c = 0; c < C::kEpiChunks; ++c) tmem_ld_32x32b_x32(t_row + 32 * c, v[c]);
        tmem_ld_wait();
        tc_fence_before_sync();
        __syncwarp();
        // The reads are complete (wait::ld): a relaxed arrive hands the
        // accumulator back without waiting for this warp's earlier D stores.
        if (lane == 0) {
          if constexpr (C::kCtaGroup == 1)
            mbar_arrive_relaxed(&acce_bar[acc]);
          else
            mbar_arrive_relaxed_cluster(acce_remote + 8u * static_cast<uint32_t>(acc));
        }
        const int row = tm * C::MMA_M + static_cast<int>(pair_rank) * C::BM + row_in_tile;
        const int col_base = tn * C::BN + half * C::kEpiCols;
        if constexpr (C::kTmaStore) {
          // One accumulator, staged stores: boxes of 32 rows x 64 bytes (32
          // bf16 or 16 f32 columns), 64B-swizzled; a chunk crossing column N
          // is stored from registers.
          const int row0 = row - static_cast<int>(lane);
          constexpr int kBoxCols = C::kStgRowBytes / (C::kBf16Out ? 2 : 4);
          constexpr int kBoxes = 32 / kBoxCols;
          const float add = epi_lean ? epi_add : 0.0f;
#pragma unroll
          for (int c = 0; c < C::kEpiChunks; ++c) {
            const int col0 = col_base + 32 * c;
            if (row0 < p.M && col0 < p.N) {
              if (!epi_lean) epilogue_general_chunk(p, col0, v[c]);
              if (col0 + 32 <= p.N) {
#pragma unroll
                for (int h = 0; h < kBoxes; ++h) {
                  if (lane == 0) bulk_wait_group_read0();
                  __syncwarp();
                  epilogue_stage_box64<C>(stg_row, lane, v[c], h, add);
                  fence_proxy_async_smem();
                  __syncwarp();
                  if (lane == 0) {
                    tma_store_2d_hint(&tmD, stg, col0 + h * kBoxCols, row0, pol_d);
                    bulk_commit_group();
                  }
                }
              } else if (row < p.M) {
                epilogue_store_chunk<C, true>(p, row, col0, v[c], add, pol_d);
              }
            }
          }
        } else if (epi_lean) {
#pragma unroll
          for (int c = 0; c < C::kEpiChunks; ++c) {
            const int col0 = col_base + 32 * c;
            if (row < p.M && col0 < p.N)
              epilogue_store_chunk<C, true>(p, row, col0, v[c], epi_add, pol_d);
          }
        } else {
#pragma unroll
          for (int c = 0; c < C::kEpiChunks; ++c) {
            const int col0 = col_base + 32 * c;
            if (row < p.M && col0 < p.N) {
              epilogue_general_chunk(p, col0, v[c]);
              epilogue_store_chunk<C, false>(p, row, col0, v[c], 0.0f, pol_d);
            }
          }
        }
      }
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // Stores still in flight finish before the block (and its shared
    // memory) goes away.
    if constexpr (C::kTmaStore)
      if (lane == 0) bulk_wait_group0();
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::kClusterCtas > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc<C::kCtaGroup>(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace tg
