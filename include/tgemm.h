/*
 * tgemm -- tiled dense contraction D = A * B^T on GB300 (sm_103a).
 *
 * C ABI of libtgemm.so.  Every entry point takes plain pointers, sizes and a
 * CUDA stream handle; no C++ or PyTorch type crosses this boundary.
 *
 * Sources for the operations (TVM TIRx documentation pages):
 *   [MMA]  "tcgen05.mma", section "Examples" -- B is stored as (N, K) and the
 *          result is a @ b.T; section "Weight-stationary and block scaling"
 *          for .block_scale with SFA/SFB.
 *   [TMA]  "cp.async.bulk.tensor", sections "Operand specification" and
 *          "Legality conditions" -- 16-byte aligned global bases, unit inner
 *          stride and suitably aligned outer byte strides; out-of-range box
 *          elements read the fill value (oob_fill 0 = zero).
 *   [LDM]  "ldmatrix / stmatrix", section "Transpose and stores" -- .trans
 *          transposes each 8x8 matrix of 16-bit elements.
 *   [EW]   "Explicit CUDA tile patterns", section "Scalar compositions", and
 *          "Tile Operands and Execution" -- an elementwise scalar function
 *          applied to each register element before the store.
 *
 * Conventions shared by every call:
 *   - Ownership: the caller allocates and owns every buffer it passes.  The
 *     library keeps its own device memory per (device, stream): a workspace
 *     (scale images of the block-scaled calls, gathered or re-pitched rows,
 *     the skinny call's f32 partial sums) and the tail split's scratch (see
 *     "Tail split").  Calls on different streams never share it; it is never
 *     shrunk and lives until process exit.  The transpose allocates nothing.
 *   - Reserved workspace (see tg_reserve_workspace): after a reservation on a
 *     stream, no call on that stream allocates device memory or synchronises
 *     anything; a call that would need more workspace than was reserved
 *     returns TG_ERR_WORKSPACE and launches nothing.
 *   - Without a reservation (the fallback), the first call on a stream that
 *     needs workspace allocates it, and a later call that needs more grows
 *     it: growing synchronises that stream (cudaStreamSynchronize), frees the
 *     old buffer and allocates a new one, so such a call may block the host.
 *     While the stream is being captured into a CUDA graph nothing is grown:
 *     the call returns TG_ERR_WORKSPACE (and the tail split is skipped).
 *     A graph captured from a stream keeps that stream's workspace addresses:
 *     do not replay it concurrently with itself or with other work on it.
 *   - The only calls that synchronise are tg_device_status,
 *     tg_reserve_workspace, the SM clock readout (tg_kernel_clock_record /
 *     _read) and, without a reservation, a call that grows its stream's
 *     workspace.
 *   - Strides are in ELEMENTS and describe row-major 2-D arrays (unit inner
 *     stride).  Pointers are device pointers and must be 16-byte aligned;
 *     every row stride times the element size must be a multiple of 16 bytes.
 *   - Execution is asynchronous on `cuda_stream` (a cudaStream_t; NULL = the
 *     legacy default stream).  A host-detectable error returns a non-zero
 *     tg_status BEFORE anything is launched.  Errors the device detects (a
 *     pipeline wait that exceeded its deadline) are reported by
 *     tg_device_status().  Nothing is thrown across the boundary and there
 *     is no CPU fallback: an unsupported request returns TG_ERR_UNSUPPORTED.
 *   - Calls on one stream are ordered; calls on different streams that share
 *     an output race, as with any CUDA kernel.
 */
#ifndef TGEMM_H
#define TGEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TG_OK = 0,
  TG_ERR_INVALID_ARG = 1, /* null pointer, negative size, stride < row length */
  TG_ERR_MISALIGNED = 2,  /* pointer or row stride violates the 16-byte rule  */
  TG_ERR_UNSUPPORTED = 3, /* valid request outside what is implemented         */
  TG_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed                 */
  TG_ERR_TIMEOUT = 5,     /* (device) a pipeline wait passed its deadline      */
  TG_ERR_NO_SCRATCH = 6,  /* problem too large for the static scratch of
                             gemm_mxfp8_blockscaled_noalloc                    */
  TG_ERR_WORKSPACE = 7    /* the stream's workspace is too small and may not
                             grow now: it is reserved, or the stream is being
                             captured into a graph                             */
} tg_status;

/* Element type of D. */
enum { TG_D_F32 = 0, TG_D_BF16 = 1 };

/* Fused elementwise epilogue, applied per element to the f32 accumulator
 * `acc` of output (i, j) before the conversion to D's type [EW]:
 *   TG_EPI_NONE           D = acc
 *   TG_EPI_ADD_SCALAR     D = acc + alpha
 *   TG_EPI_SILU_AFFINE    D = silu(acc) * alpha + beta      (the pages' silu_affine)
 *   TG_EPI_BIAS_COL       D = acc + bias[j]
 *   TG_EPI_BIAS_COL_SILU  D = silu(acc + bias[j])
 *   TG_EPI_AFFINE         D = acc * alpha + beta            (e.g. a per-tensor scale)
 * with silu(x) = x / (1 + exp(-x)) evaluated in f32 (CUDA expf). */
enum {
  TG_EPI_NONE = 0,
  TG_EPI_ADD_SCALAR = 1,
  TG_EPI_SILU_AFFINE = 2,
  TG_EPI_BIAS_COL = 3,
  TG_EPI_BIAS_COL_SILU = 4,
  TG_EPI_AFFINE = 5
};

/* Epilogue description for the *_ex entry points (caller-owned, read during
 * the call only).  bias: device f32 [N], 16-byte aligned, used by the
 * BIAS_COL ops only (NULL otherwise); alpha/beta as in the table above. */
typedef struct tg_epilogue {
  int op;
  float alpha;
  float beta;
  const float* bias;
} tg_epilogue;

/*
 * Tail split.  The GEMM kernels are persistent: every SM (or SM pair) walks
 * its share of the output tiles.  When the R tiles of a dense (bf16)
 * product's last wave (after W >= 0 full waves over all co-resident units)
 * fill at most half of the units, each of them is cut into S pieces along K
 * (S <= 4, S * R <= the units, pieces of >= 4 stages) that run at the same time;
 * every piece writes its f32 partial tile into a per-(device, stream)
 * scratch of 20 MiB and arrives on a counter; the piece whose arrival
 * completes the count adds the S partials in piece order and stores D.  No
 * piece waits for another, so the call completes however many of its CTAs
 * are resident at once (e.g. beside kernels on other streams).  The scratch
 * is allocated by tg_reserve_workspace, or else with cudaMalloc on the first
 * call that splits on a stream (a stream being captured runs unsplit
 * instead).  Results agree with the unsplit product within the tolerances
 * above; the partials are added in a fixed order, so repeated calls give
 * identical bits.
 */

/*
 * Result bits.  Each output tile accumulates its K range in an order fixed
 * by the persistent schedule: forwards, or backwards in every other wave of
 * tiles (which keeps the K slices a unit needs next in L2), and split into
 * pieces in a tail split.  The same call (shape, flags, strides, device)
 * therefore always returns the same bits; calls with other flags, or on a
 * device with another SM count, may differ in the last bits, within the
 * tolerances.  Exact inputs (every partial sum representable) give the exact
 * result whatever the order.
 */

/* Launch flags (bit set). */
enum {
  TG_FLAG_CTA_PAIR = 1u, /* cta_group::2: two CTAs of a cluster share one
                            256-row MMA; each loads half of the B tile      */
  TG_FLAG_MULTICAST = 2u, /* clusters of two MMA units on vertically adjacent
                            tiles share the B tile by TMA multicast.  With
                            TG_FLAG_CTA_PAIR: two pairs (each CTA loads a
                            quarter of B); measured 2-3% slower than plain
                            pairs at 8192^3, so off by default.  Alone (bf16
                            only): two single CTAs, each loading half of B;
                            gemm_bf16 with flags 0 picks these by itself for
                            K <= 1536 with M, N >= 3000, where they measured
                            6-30% faster (slower at K >= 2048).  Results
                            agree within the tolerances either way (see
                            "Result bits" below).  Multicast clusters (asked
                            for or chosen) run only when A and B (and the
                            scale arrays) are allocations of the current
                            device (cudaPointerGetAttributes); for host,
                            managed or another GPU's memory the call runs
                            the plain kernel instead.  This library is
                            single-GPU code: one process drives one GPU.     */
  TG_FLAG_GATHER_TMA = 4u /* gemm_bf16_gather only: load the gathered A rows
                            inside the GEMM with TMA tile::gather4 instead
                            of copying them into the workspace first.
                            Results agree within the tolerances; slower on
                            large shapes (see there).                       */
};

/*
 * gemm_bf16 -- D[M,N] = A[M,K] * B[N,K]^T (+ epilogue), bf16 inputs, f32
 * accumulation in tensor memory [MMA].
 *   A    : device, bf16 [M, K], row stride lda (elements), K-major.
 *   B    : device, bf16 [N, K], row stride ldb, K-major.
 *   D    : device, [M, N] of d_dtype (TG_D_F32 or TG_D_BF16), row stride ldd.
 *   M,N,K: sizes, 0 <= M, N, K < 2^31.  M or N == 0: nothing is launched.
 *          K == 0: D = epilogue(0).  Any size need not be a tile multiple:
 *          loads past the edge read zeros [TMA], stores past it are dropped.
 *   epilogue, epi_scalar: TG_EPI_NONE, or TG_EPI_ADD_SCALAR with constant s
 *          (the other epilogues need gemm_bf16_ex).
 *   flags: 0, TG_FLAG_CTA_PAIR, TG_FLAG_MULTICAST (single-CTA clusters), or
 *          TG_FLAG_CTA_PAIR | TG_FLAG_MULTICAST.
 * Rounding: f32 -> bf16 D is round-to-nearest-even.  Alignment: A, B, D
 * 16-byte aligned; lda*2, ldb*2, ldd*sizeof(D) multiples of 16.
 * Re-pitch: when lda*2 (or ldb*2) is not a multiple of 32 (rows only 16-byte
 * aligned) and the product is large against its operands (M*N/(M+N) >=
 * 1250), that operand is first copied into the stream's library workspace
 * at a 128-byte pitch (ceil(K/64)*64 elements per row; K elements read per
 * row); the result is the same, bit for bit.  Multicast clusters of CTA
 * pairs (TG_FLAG_CTA_PAIR | TG_FLAG_MULTICAST over this device's memory)
 * read such rows in place: with half as many B loads the copy no longer
 * pays there.
 * Returns TG_OK once the kernel is enqueued, else an error (nothing enqueued).
 */
int gemm_bf16(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
              int64_t M, int64_t N, int64_t K, int d_dtype, int epilogue, float epi_scalar,
              unsigned flags, void* cuda_stream);

/*
 * gemm_bf16_ex -- gemm_bf16 with a full epilogue description.  epi may be
 * NULL (D = acc).  An unknown op, or a BIAS_COL op without a bias vector,
 * returns TG_ERR_INVALID_ARG; a bias not 16-byte aligned TG_ERR_MISALIGNED.
 * gemm_bf16(..., epilogue, s, ...) equals gemm_bf16_ex with {epilogue, s, 0,
 * NULL} and accepts only TG_EPI_NONE and TG_EPI_ADD_SCALAR.
 */
int gemm_bf16_ex(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
                 int64_t M, int64_t N, int64_t K, int d_dtype, const tg_epilogue* epi,
                 unsigned flags, void* cuda_stream);

/*
 * gemm_mxfp8_blockscaled -- block-scaled MXFP8 product [MMA, .block_scale]:
 *   D[i,j] = sum_k (A[i,k] * 2^(SFA[i,k/32]-127)) * (B[j,k] * 2^(SFB[j,k/32]-127))
 *   A   : device, FP8 E4M3FN bytes [M, K], row stride lda (bytes).
 *   B   : device, FP8 E4M3FN bytes [N, K], row stride ldb.
 *   SFA : device, E8M0 bytes [M, K/32], row stride ld_sfa (any value >= K/32).
 *   SFB : device, E8M0 bytes [N, K/32], row stride ld_sfb.
 *   D, ldd, d_dtype, epilogue, epi_scalar, flags: as for gemm_bf16, except
 *   that TG_FLAG_MULTICAST needs TG_FLAG_CTA_PAIR (alone: TG_ERR_INVALID_ARG).
 *   K must be a multiple of 32 (one scale per 32 K elements); otherwise
 *   TG_ERR_INVALID_ARG.  lda and ldb must be multiples of 16.
 * The scales are first rearranged on the device into the tensor-memory image
 * the MMA reads (row r -> lane r%32, byte column 4*(r/32)) in the stream's
 * library workspace (ceil(M/128)*ceil(K/128)*512 + ceil(N/128)*
 * ceil(K/128)*512 bytes).
 */
int gemm_mxfp8_blockscaled(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           int epilogue, float epi_scalar, unsigned flags, void* cuda_stream);

/* gemm_mxfp8_blockscaled_ex -- gemm_mxfp8_blockscaled with a full epilogue
 * description (as gemm_bf16_ex). */
int gemm_mxfp8_blockscaled_ex(const void* A, int64_t lda, const void* B, int64_t ldb,
                              const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                              void* D, int64_t ldd, int64_t M, int64_t N, int64_t K,
                              int d_dtype, const tg_epilogue* epi, unsigned flags,
                              void* cuda_stream);

/*
 * gemm_bf16_skinny -- gemm_bf16_ex for few rows (1 <= M <= 128), where reading
 * B once from HBM bounds the product.  The operands are swapped so that 128
 * rows of B fill the MMA's M side and the M rows of A its N side (rounded up
 * to 16, 32, 64 or 128); every 128-row tile of B is split into split_k pieces
 * of K (0: chosen from N, K and the SM count) whose f32 partial tiles are
 * added into the result with TMA reduce-add ["cp.async.bulk.tensor",
 * reductions].  D, ldd, d_dtype, epi: as for gemm_bf16_ex.
 *   M > 128: TG_ERR_UNSUPPORTED; split_k < 0: TG_ERR_INVALID_ARG.
 * With more than one piece the partial sums are added in a run-dependent
 * order, so the last bits of D may differ between runs.  bf16 D, and f32 D
 * with a SiLU epilogue, take one extra elementwise pass, and so does f32 D
 * with N % 4 != 0; those cases use the stream's library workspace
 * (M * ceil(N/4)*4 * 4 bytes).
 */
int gemm_bf16_skinny(const void* A, int64_t lda, const void* B, int64_t ldb, void* D, int64_t ldd,
                     int64_t M, int64_t N, int64_t K, int d_dtype, const tg_epilogue* epi,
                     int split_k, void* cuda_stream);

/*
 * gemm_bf16_gather -- bf16 GEMM over gathered rows of A (a mixture-of-experts
 * layer's tokens for one expert): D[i, :] = A[row_idx[i], :] * B^T (+ epi)
 * for 0 <= i < M [MMA; TMA tile::gather4 loads of the A tile].
 *   A       : device, bf16 [a_rows, K], row stride lda (elements).
 *   row_idx : device, int32 [M]; any row of A, in any order, repeats allowed.
 *             An index outside [0, a_rows) gives a zero row (D = epi(0)).
 *   B, ldb, D, ldd, N, K, d_dtype, epi: as for gemm_bf16_ex; D is [M, N].
 *   flags   : TG_FLAG_CTA_PAIR and / or TG_FLAG_GATHER_TMA (TG_FLAG_MULTICAST:
 *             TG_ERR_UNSUPPORTED).
 *   K > 0 with a NULL row_idx or a_rows == 0: TG_ERR_INVALID_ARG.
 * By default the rows are first gathered into the stream's library
 * workspace (M * ceil(K/64)*64 * 2 bytes: rows at a 128-byte pitch) and the
 * dense kernel runs on them.  With
 * TG_FLAG_GATHER_TMA the GEMM loads them itself with tile::gather4 (no
 * workspace); that issue rate bounds it at ~60% of the dense kernel for
 * 4096 x 8192 x 8192.
 */
int gemm_bf16_gather(const void* A, int64_t lda, int64_t a_rows, const int32_t* row_idx,
                     int64_t M, const void* B, int64_t ldb, void* D, int64_t ldd, int64_t N,
                     int64_t K, int d_dtype, const tg_epilogue* epi, unsigned flags,
                     void* cuda_stream);

/* tg_gemm_tail_split -- the number of K pieces (1: none) into which
 * gemm_bf16 cuts each tile for this shape on the current device (flags: 0 or
 * TG_FLAG_CTA_PAIR), for operands in the current device's memory (a stream
 * being captured without tail scratch runs unsplit); minus a status code on
 * failure.  See "Tail split". */
int tg_gemm_tail_split(int64_t M, int64_t N, int64_t K, unsigned flags);

/* tg_gemm_multicast -- 1 if gemm_bf16 / gemm_bf16_ex with these operands,
 * sizes and flags (0, TG_FLAG_CTA_PAIR, TG_FLAG_MULTICAST or both) run
 * multicast clusters, 0 if they run the plain kernel (in particular when A or
 * B is not an allocation of the current device, or that cannot be told);
 * minus a status code for invalid arguments.  Reads pointer attributes only:
 * nothing is launched or dereferenced. */
int tg_gemm_multicast(const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                      unsigned flags);

/* Call kinds for tg_workspace_bytes. */
enum {
  TG_CALL_GEMM_BF16 = 0,        /* gemm_bf16, gemm_bf16_ex                     */
  TG_CALL_GEMM_MXFP8 = 1,       /* gemm_mxfp8_blockscaled(_ex)                 */
  TG_CALL_GEMM_MXFP4 = 2,       /* gemm_mxfp4_blockscaled                      */
  TG_CALL_GEMM_NVFP4 = 3,       /* gemm_nvfp4_blockscaled                      */
  TG_CALL_GEMM_BF16_SKINNY = 4, /* gemm_bf16_skinny                            */
  TG_CALL_GEMM_BF16_GATHER = 5  /* gemm_bf16_gather (M = gathered rows)        */
};

/*
 * tg_workspace_bytes -- bytes of stream workspace one call of kind `call`
 * needs for these sizes: lda, ldb (elements, as passed to the call; used by
 * the bf16 re-pitch rule), d_dtype and epi_op (used by the skinny call) and
 * flags (TG_FLAG_CTA_PAIR; TG_FLAG_GATHER_TMA for the gather call).  Calls on
 * one stream run in order and reuse the workspace from its start, so a
 * stream needs the maximum over its calls, not the sum.  The tail split's
 * scratch is separate (tg_reserve_workspace always adds it).  Minus a status
 * code for invalid arguments.  Host arithmetic only: no CUDA call.
 */
int64_t tg_workspace_bytes(int call, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                           int d_dtype, int epi_op, unsigned flags);

/*
 * tg_reserve_workspace -- allocate now, for the current device and
 * `cuda_stream`, a workspace of at least `bytes` (e.g. the maximum of
 * tg_workspace_bytes over the calls the stream will make) and the tail
 * split's scratch, then mark the stream reserved: from then on no call on
 * it allocates device memory or synchronises, and one needing more workspace
 * returns TG_ERR_WORKSPACE.  May be called again to grow the reservation.
 * Synchronises the stream.  TG_ERR_WORKSPACE while the stream is being
 * captured; TG_ERR_CUDA if an allocation fails; TG_ERR_INVALID_ARG for
 * bytes < 0.
 */
int tg_reserve_workspace(void* cuda_stream, int64_t bytes);

/* Number of device allocations (cudaMalloc) the library has made since it
 * was loaded, over all devices and streams: workspace and tail scratch.  A
 * caller can check that a code section allocated nothing. */
uint64_t tg_workspace_alloc_count(void);

/* tg_gemm_repitch -- which operands gemm_bf16 / gemm_bf16_ex re-pitch for
 * this shape, these row strides and these flags (see gemm_bf16), for
 * operands in the current device's memory: bit 0 A, bit 1 B (0: neither);
 * minus TG_ERR_INVALID_ARG for negative sizes or flags other than
 * TG_FLAG_CTA_PAIR / TG_FLAG_MULTICAST.  Host arithmetic only: no CUDA call,
 * no device needed. */
int tg_gemm_repitch(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, unsigned flags);

/* tg_skinny_split_count -- the number of K pieces gemm_bf16_skinny uses for
 * (N, K, split_k) on the current device, or minus a status code. */
int tg_skinny_split_count(int64_t N, int64_t K, int split_k);

/*
 * gemm_mxfp4_blockscaled -- block-scaled FP4 product with MX scales
 * [MMA, .kind::mxf4nvf4 .block_scale .scale_vec::2X]:
 *   D[i,j] = sum_k (a[i,k] * 2^(SFA[i,k/32]-127)) * (b[j,k] * 2^(SFB[j,k/32]-127))
 *   A   : device, packed FP4 E2M1 [M, K/2] bytes, row stride lda (bytes):
 *         element k of a row is the low nibble of byte k/2 for even k and
 *         the high nibble for odd k.
 *   B   : device, packed E2M1 [N, K/2] bytes, row stride ldb (bytes).
 *   SFA : device, E8M0 bytes [M, K/32], row stride ld_sfa (>= K/32).
 *   SFB : device, E8M0 bytes [N, K/32], row stride ld_sfb.
 *   D, ldd, d_dtype, epi: as for gemm_bf16_ex.  flags: 0 or TG_FLAG_CTA_PAIR
 *   (TG_FLAG_MULTICAST: TG_ERR_UNSUPPORTED with a pair, else TG_ERR_INVALID_ARG).
 *   K must be a multiple of 32; otherwise TG_ERR_INVALID_ARG.  lda >= K/2,
 *   ldb >= K/2, both multiples of 16 (TG_ERR_MISALIGNED).
 * The scales are rearranged into the tensor-memory image in the stream's
 * library workspace, as for gemm_mxfp8_blockscaled (two 512-byte images per
 * 128 rows and 256 K).
 */
int gemm_mxfp4_blockscaled(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           const tg_epilogue* epi, unsigned flags, void* cuda_stream);

/*
 * gemm_nvfp4_blockscaled -- block-scaled FP4 product with UE4M3 scales per
 * 16 elements [MMA, .kind::mxf4nvf4 .block_scale .scale_vec::4X]:
 *   D[i,j] = sum_k (a[i,k] * ue4m3(SFA[i,k/16])) * (b[j,k] * ue4m3(SFB[j,k/16]))
 *   A, B: packed E2M1 as for gemm_mxfp4_blockscaled.
 *   SFA : device, UE4M3 bytes [M, K/16] (E4M3 with the sign bit clear; a set
 *         sign bit or 0x7F is not a valid scale), row stride ld_sfa >= K/16.
 *   SFB : device, UE4M3 bytes [N, K/16], row stride ld_sfb.
 *   K must be a multiple of 16; otherwise TG_ERR_INVALID_ARG.  A per-tensor
 *   scale (the second level of NVFP4 scaling) is applied with TG_EPI_AFFINE.
 * Workspace: four 512-byte images per 128 rows and 256 K.
 */
int gemm_nvfp4_blockscaled(const void* A, int64_t lda, const void* B, int64_t ldb,
                           const void* SFA, int64_t ld_sfa, const void* SFB, int64_t ld_sfb,
                           void* D, int64_t ldd, int64_t M, int64_t N, int64_t K, int d_dtype,
                           const tg_epilogue* epi, unsigned flags, void* cuda_stream);

/*
 * gemm_mxfp8_blockscaled_noalloc -- the same product as gemm_mxfp8_blockscaled,
 * for callers that must not allocate device memory (a host framework whose
 * own pool owns the device memory, a latency-bound serving loop where
 * cudaMalloc/cudaFree would synchronise the device, a deployment that
 * forbids allocation after start-up).  The pages have no counterpart: this
 * is a library-usage variant, not part of the method.
 *   Arguments, layouts, alignment rules and results: as gemm_mxfp8_blockscaled.
 *   Scratch: a fixed 8 MiB device array inside the library (reserved on every
 *   GPU that loads it, until the process exits) instead of the allocated
 *   workspace.  The call never calls cudaMalloc or cudaFree.  A problem needs
 *   (ceil(M/r)*(r/128) + 2*ceil(N/256)) * ceil(K/128) * 512 bytes of it, with
 *   r = 256 under TG_FLAG_CTA_PAIR and 128 otherwise (4 MiB at 8192^3);
 *   larger problems return TG_ERR_NO_SCRATCH and launch nothing.
 *   Sharing: every call on a device uses the same array.  Calls whose kernels
 *   may overlap on the GPU (unordered streams) race on it.  Each call rewrites
 *   all scratch it reads, so leftover contents from an earlier call are harmless.
 *   Set-up: the first call on each device looks up the array's device address
 *   with that device current; make that first call before any stream capture.
 */
int gemm_mxfp8_blockscaled_noalloc(const void* A, int64_t lda, const void* B, int64_t ldb,
                                   const void* SFA, int64_t ld_sfa, const void* SFB,
                                   int64_t ld_sfb, void* D, int64_t ldd, int64_t M, int64_t N,
                                   int64_t K, int d_dtype, int epilogue, float epi_scalar,
                                   unsigned flags, void* cuda_stream);

/*
 * tile_transpose_b16 -- out[j,i] = in[i,j] for 16-bit elements, bit-exact
 * (raw bit patterns, NaNs included) [LDM].  Built from ldmatrix.trans and
 * stmatrix through shared memory.
 *   in  : device, [rows, cols] 16-bit, row stride ld_in (elements).
 *   out : device, [cols, rows] 16-bit, row stride ld_out.  Must not overlap in.
 *   rows, cols >= 0 (0: nothing launched).  Pointers 16-byte aligned;
 *   ld_in and ld_out multiples of 8.
 */
int tile_transpose_b16(const void* in, int64_t ld_in, void* out, int64_t ld_out, int64_t rows,
                       int64_t cols, void* cuda_stream);

/*
 * tg_device_status -- synchronise `cuda_stream`, then return and clear the
 * current device's status word: TG_OK, or TG_ERR_TIMEOUT when a kernel's
 * pipeline wait passed its deadline (the kernel then stopped early, left its
 * outputs incomplete and released its tensor memory), or TG_ERR_CUDA when
 * the synchronisation itself failed.  `site` (may be NULL) receives the code
 * of the wait that expired.  After an error it also clears the library's
 * tail-split counters on this device (see "Tail split" above); other streams of
 * the device should be idle at that point.
 */
int tg_device_status(void* cuda_stream, uint32_t* site);

/*
 * SM clock of the GEMM kernels.  NVML (nvidia-smi) can report the maximum SM
 * clock while a power-capped tensor kernel actually runs several hundred MHz
 * lower, and a kernel's fraction of the tensor pipe's peak depends on that
 * clock.  While recording is on, every MMA unit (a CTA, or the leading CTA
 * of a pair) of each gemm_* launch on the current device adds the SM cycles
 * and nanoseconds (%clock64, %globaltimer) between the start and the end of
 * its MMA issue into a sum kept per kind; the readout is their ratio.
 *
 * tg_kernel_clock_record -- enable != 0: clear the sums and record the
 *   launches made after this call; 0: stop recording (the sums are kept).
 *   Synchronises the device.  The skinny GEMM and the transpose do not record.
 *   A launch captured into a CUDA graph while recording is on keeps adding
 *   whenever the graph is replayed, also after recording was stopped.
 * tg_kernel_clock_read -- the average SM clock in MHz (0 if nothing was
 *   recorded) of the launches of `kind` since recording was last enabled,
 *   and the number of MMA units that contributed (`units` may be NULL).
 *   Synchronises the device.  TG_ERR_INVALID_ARG for an unknown kind or a
 *   NULL `mhz`.  Not on the pages: a measurement aid.
 */
enum {
  TG_CLOCK_BF16 = 0,   /* gemm_bf16, gemm_bf16_ex, gemm_bf16_gather */
  TG_CLOCK_MXFP8 = 1,  /* gemm_mxfp8_blockscaled(_ex, _noalloc)     */
  TG_CLOCK_MXFP4 = 2,  /* gemm_mxfp4_blockscaled                    */
  TG_CLOCK_NVFP4 = 3   /* gemm_nvfp4_blockscaled                    */
};
int tg_kernel_clock_record(int enable);
int tg_kernel_clock_read(int kind, double* mhz, uint64_t* units);

/* Deadline of every bounded pipeline wait, in nanoseconds (default 2e9).
 * Applies to launches made after the call; 0 is rejected. */
int tg_set_wait_timeout_ns(uint64_t ns);

/* Static string for a tg_status value. */
const char* tg_status_string(int status);

/* The cudaError_t behind the most recent TG_ERR_CUDA returned on this thread. */
int tg_last_cuda_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int tg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_H */
