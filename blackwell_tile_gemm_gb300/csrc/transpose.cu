// tile_transpose_b16: out[j, i] = in[i, j] on raw 16-bit patterns.
//
// Built from the data-movement instructions of "ldmatrix / stmatrix" (TVM TIRx
// tile-operation guide): .trans transposes each 8x8 matrix of 16-bit
// elements (section "Transpose and stores": register element (row, 2w+h)
// comes from shared element (2w+h, row), owned by lane 4*row + w), and
// stmatrix writes a register image back to the rows its address providers
// name (lane 8*matrix + row supplies that row's address).
//
// Each CTA moves one 64 x 64 tile:
//   1. ld.global.v4 (16-byte rows of 8 elements) -> shared tile S, where the
//      16-byte chunk c of row r is stored at chunk c ^ (r % 8) so that the 8
//      rows an ldmatrix phase touches fall in 8 different bank groups;
//   2. per warp, two ldmatrix.x4.trans of S blocks (8w, 8c) -> registers now
//      hold the transposed 8x8 blocks -> stmatrix.x4 into the output tile T at
//      block (8c, 8w), with the same chunk swizzle;
//   3. ld.shared.v4 rows of T -> st.global.v4 into out.
// Edge tiles fall back to 16-bit loads / stores for the partial chunks.
#include <cstdint>

#include <cuda_runtime.h>

#include "tg_internal.h"
#include "tg_ptx.cuh"

namespace tg {

namespace {

constexpr int kTile = 64;
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t chunk_offset(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(kThreads)
    transpose_b16_kernel(const uint16_t* __restrict__ in, int64_t ld_in,
                         uint16_t* __restrict__ out, int64_t ld_out, int rows, int cols,
                         int tiles_c) {
  __shared__ __align__(128) uint8_t S[kTile * kTile * 2];
  __shared__ __align__(128) uint8_t T[kTile * kTile * 2];
  const int tile = blockIdx.x;
  const int i0 = (tile / tiles_c) * kTile;   // input rows
  const int j0 = (tile % tiles_c) * kTile;   // input columns
  const int tid = threadIdx.x;
  const bool full = (i0 + kTile <= rows) && (j0 + kTile <= cols);

  // 1. global -> S
  uint4 v[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int c = tid + q * kThreads;
    const int r = c >> 3, ch = c & 7;
    const int i = i0 + r, j = j0 + ch * 8;
    if (full) {
      v[q] = ld_global_nc_v4(in + static_cast<int64_t>(i) * ld_in + j);
    } else {
      uint32_t w[4] = {0, 0, 0, 0};
      if (i < rows) {
        const uint16_t* src = in + static_cast<int64_t>(i) * ld_in;
        if (j + 8 <= cols) {
          const uint4 t = ld_global_nc_v4(src + j);
          w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (j + e < cols) w[e >> 1] |= static_cast<uint32_t>(src[j + e]) << (16 * (e & 1));
        }
      }
      v[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int c = tid + q * kThreads;
    *reinterpret_cast<uint4*>(S + chunk_offset(c >> 3, c & 7)) = v[q];
  }
  __syncthreads();

  // 2. S -> registers (ldmatrix.trans) -> T (stmatrix)
  {
    const int w = tid >> 5;             // S block row (8 input rows)
    const int lane = tid & 31;
    const int m = lane >> 3, rr = lane & 7;
    const uint32_t sS = smem_addr(S), sT = smem_addr(T);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ch = 4 * h + m;         // S block column = T block row
      uint32_t r0, r1, r2, r3;
      ldmatrix_x4_trans(sS + chunk_offset(8 * w + rr, ch), r0, r1, r2, r3);
      stmatrix_x4(sT + chunk_offset(8 * ch + rr, w), r0, r1, r2, r3);
    }
  }
  __syncthreads();

  // 3. T -> global
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int c = tid + q * kThreads;
    const int t = c >> 3, ch = c & 7;
    const int oj = j0 + t, oi = i0 + ch * 8;
    const uint4 x = *reinterpret_cast<const uint4*>(T + chunk_offset(t, ch));
    if (full) {
      st_global_v4(out + static_cast<int64_t>(oj) * ld_out + oi, x.x, x.y, x.z, x.w);
    } else if (oj < cols) {
      uint16_t* dst = out + static_cast<int64_t>(oj) * ld_out;
      if (oi + 8 <= rows) {
        st_global_v4(dst + oi, x.x, x.y, x.z, x.w);
      } else {
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (oi + e < rows) dst[oi + e] = static_cast<uint16_t>(w4[e >> 1] >> (16 * (e & 1)));
      }
    }
  }
}

}  // namespace

int launch_transpose_b16(const void* in, int64_t ld_in, void* out, int64_t ld_out, int64_t rows,
                         int64_t cols, cudaStream_t stream, DeviceCtx* ctx) {
  (void)ctx;
  const int64_t tiles_r = (rows + kTile - 1) / kTile;
  const int64_t tiles_c = (cols + kTile - 1) / kTile;
  const int64_t tiles = tiles_r * tiles_c;
  if (tiles > 0x7FFFFFFF) return TG_ERR_UNSUPPORTED;
  transpose_b16_kernel<<<static_cast<unsigned>(tiles), kThreads, 0, stream>>>(
      static_cast<const uint16_t*>(in), ld_in, static_cast<uint16_t*>(out), ld_out,
      static_cast<int>(rows), static_cast<int>(cols), static_cast<int>(tiles_c));
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? TG_OK : cuda_fail(e);
}

}  // namespace tg
