/*
 * tgemm probes -- small single-CTA kernels that run the pages' worked
 * examples and dump raw hardware mappings, so that each building block of
 * the GEMM and transpose path can be checked on its own against the CPU
 * oracle.  They are part of libtgemm.so; they are not on the GEMM path.
 *
 * All pointers are device pointers owned by the caller; every call is
 * asynchronous on `cuda_stream` and returns a tg_status (tgemm.h) before
 * launching anything if an argument is wrong.
 */
#ifndef TGEMM_PROBES_H
#define TGEMM_PROBES_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* "Tile Operands and Execution", section "A Load, Compute, and Store
 * Example": 64 threads, each loads twelve f32 with three ld.global.v4.b32,
 * adds one, stores with st.global.v4.b32.  a, b: f32 [2, 32, 3, 4], 16-byte
 * aligned. */
int tg_probe_add_one_v4(const float* a, float* b, void* cuda_stream);

/* "ldmatrix / stmatrix", section "Example: interleaved shared rows and
 * register slots 0, 2, 8, 10": x: uint32 [16, 4, 2] is placed in shared
 * memory with strides (8, 1, 128) words; every lane fills twelve registers
 * with 4294966519 and issues two ldmatrix .x2 on the (k, m, r, w) view
 * SM[2r+m, w, k]; out: uint32 [32, 12] receives each lane's registers. */
int tg_probe_ldmatrix_x2_interleaved(const uint32_t* x, uint32_t* out, void* cuda_stream);

/* ldmatrix.m8n8.x{n}[.trans].shared.b16 of n matrices stored as rows:
 * smem_image: uint16 [n, 8, 8] (matrix, row, column); out: uint32 [32, n],
 * word i of lane l.  n in {1, 2, 4}, trans in {0, 1}. */
int tg_probe_ldmatrix(const uint16_t* smem_image, int n, int trans, uint32_t* out,
                      void* cuda_stream);

/* stmatrix.m8n8.x{n}[.trans].shared.b16: regs: uint32 [32, n] (word i of
 * lane l); out: uint16 [n, 8, 8], the shared rows written. */
int tg_probe_stmatrix(const uint32_t* regs, int n, int trans, uint16_t* out, void* cuda_stream);

/* "cp.async.bulk.tensor", section "Example: two explicit 8x16 boxes": one
 * lane loads a (16, 16) uint32 tensor as two 8x16 TMA boxes at (0, 0) and
 * (8, 0) on one barrier phase expecting 1024 bytes.  a, out: uint32 [16, 16]. */
int tg_probe_tma_two_boxes(const uint32_t* a, uint32_t* out, void* cuda_stream);

/* One TMA load of a bf16 [rows, 64] box with 128-byte swizzle; out receives
 * the raw shared-memory bytes (rows * 128).  rows in 8..256, multiple of 8. */
int tg_probe_tma_swizzle128(const uint16_t* src, int rows, uint8_t* out, void* cuda_stream);

/* "tcgen05.mma", section "Example: four K16 issues for a 128x64x64 product",
 * in bf16: a: bf16 [128, 64] and b: bf16 [64, 64] (B stored as (N, K)) are
 * written to 128-byte-swizzled K-major shared layouts with ordinary stores,
 * one thread issues four kind::f16 M128 N64 K16 MMAs and one commit, four
 * warps read TMEM back with tcgen05.ld 32x32b; out: f32 [128, 64] = a @ b.T. */
int tg_probe_mma_128x64x64(const uint16_t* a, const uint16_t* b, float* out, void* cuda_stream);

/* The same example with the weight-stationary opcode ("tcgen05.mma": M128
 * .ws uses TMEM layout D like M128 without .ws; CTA group 1, N = 64):
 * tcgen05.mma.ws.cta_group::1.kind::f16, same operands and read-back. */
int tg_probe_mma_ws_128x64x64(const uint16_t* a, const uint16_t* b, float* out,
                              void* cuda_stream);

/* "Explicit CUDA tile patterns", section "TMEM transfers": one CTA of four
 * warps writes row * 256 + column into TMEM rows 0..127, columns 0..31
 * (tcgen05.st 32x32b; row = 32 * warp + lane), then reads columns 0..15 back
 * with tcgen05.ld 16x64b.x8, 16x128b.x4, 16x256b.x2, 32x32b.x8 and
 * 16x32bx2.x8 (imm_half_splitoff = (16 << 16) + 8), the 16-lane shapes at
 * each warp's first lane.  out: device uint32 [5 shapes][128 threads][8
 * registers]. */
int tg_probe_tmem_shapes(uint32_t* out, void* cuda_stream);

/* Tensor-pipe rate with no memory traffic: `ctas` CTAs (one per SM when
 * ctas <= SM count), each issuing iters x 4 back-to-back M128 N256 MMAs on
 * fixed shared-memory operands into one TMEM accumulator.  kind: 0 = bf16
 * kind::f16 K16, 1 = E4M3 kind::mxf8f6f4.block_scale K32 (unit scales),
 * 2 = E4M3 kind::f8f6f4 K32, 3 = packed E2M1 kind::mxf4nvf4.block_scale
 * .scale_vec::2X K64 (unit E8M0 scales), 4 = the same with .scale_vec::4X
 * (unit UE4M3 scales).  cycles: device uint64 [2*ctas]; per CTA, SM
 * clock cycles and then nanoseconds from the first issue to completion of
 * the last MMA.  Each CTA gets an SM of its own.  Dense
 * FLOP per SM per cycle = 2*128*256*K*4*iters / cycles.  This is the
 * "tensor-pipe peak" denominator; the pages publish no rate. */
int tg_probe_mma_rate(int kind, int iters, int ctas, unsigned long long* cycles,
                      void* cuda_stream);

/* Occupies SMs: `blocks` (1..4096) blocks of one warp, each with 200 KB of
 * dynamic shared memory (so that no GEMM CTA fits beside it), sleep until
 * `ns` (1..10^9) nanoseconds have passed.  Used to show that a GEMM launched
 * meanwhile on another stream completes while only some of its CTAs can be
 * resident.  Not part of the contraction: a test aid. */
int tg_probe_hold_sms(int blocks, uint64_t ns, void* cuda_stream);

/* Waits on an mbarrier that nothing completes, with deadline `timeout_ns`
 * (1..10^9); the bounded wait gives up and records TG_ERR_TIMEOUT with site
 * code 99 in the status word that tg_device_status() returns. */
int tg_probe_wait_timeout(uint64_t timeout_ns, void* cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* TGEMM_PROBES_H */
