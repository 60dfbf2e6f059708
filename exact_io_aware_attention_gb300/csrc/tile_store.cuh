// Epilogue helper shared by the kernels: one thread's row of an fp32
// accumulator in tensor memory leaves through shared memory and TMA.
#pragma once

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

// Row r of a 128-row tile: kCols fp32 columns (a multiple of 32) read from
// tensor memory at `tacc` (this warp's lane quadrant already in the address),
// times `sc`, rounded to the 16-bit type (kF16: f16, else bf16) and written
// to shared memory at `s_tile` as 64-column chunks of 128 rows x 128 bytes in
// the 128-byte swizzle of the tensor maps; then lane 0 of the warp stores its
// 32 rows through `tm` (a map with 64 x 32 boxes) at columns x0.. and rows
// tile_row0 + ... of head (h_idx, b_idx). Columns at or past `d_cols` are
// neither read nor stored, and the map clips rows at or past the tensor's row
// count and columns past its width (a last chunk of 32 columns stores 64, of
// which the map writes the first 32); a warp whose first row is at or past
// `n_rows` stores nothing. With any == false the row is zero.
//
// Every thread of the warp must call it (tensor-memory loads are warp-wide),
// and the buffer at s_tile must be free: no MMA or copy still reads it.
// store_rows_tma is a function of its own, called once per CTA, so that its
// registers do not weigh on the kernels' main loops; store_rows_tma_inl is the
// same code inlined, for kernels whose warpgroups set their own register
// counts (setmaxnreg), where every call is inlined.
template <int kCols, bool kF16>
__device__ __forceinline__ void store_rows_tma_inl(const CUtensorMap *tm, uint32_t tacc,
                                            uint32_t s_tile, int r, int tile_row0, int x0,
                                            float sc, bool any, int d_cols, int n_rows,
                                            int h_idx, int b_idx) {
  static_assert(kCols % 32 == 0, "whole 32-column groups");
  constexpr uint32_t kChunkBytes = kTile * 128;
#pragma unroll
  for (int q = 0; q < kCols / 32; ++q) {
    if (x0 + q * 32 >= d_cols) break;
    uint32_t o[32];
    if (any) {
      tmem_ld32(tacc + q * 32, o);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int x = 0; x < 32; ++x) o[x] = 0u;
    }
    const uint32_t rowbase = s_tile + (q >> 1) * kChunkBytes + r * 128;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const uint32_t piece = uint32_t((q & 1) * 4 + x) ^ uint32_t(r & 7);
      st_shared_v4(rowbase + (piece << 4),
                   pack2<kF16>(__uint_as_float(o[8 * x + 0]) * sc, __uint_as_float(o[8 * x + 1]) * sc),
                   pack2<kF16>(__uint_as_float(o[8 * x + 2]) * sc, __uint_as_float(o[8 * x + 3]) * sc),
                   pack2<kF16>(__uint_as_float(o[8 * x + 4]) * sc, __uint_as_float(o[8 * x + 5]) * sc),
                   pack2<kF16>(__uint_as_float(o[8 * x + 6]) * sc, __uint_as_float(o[8 * x + 7]) * sc));
    }
  }
  const int warp_row = (r & (kTile - 1)) & ~31;  // this warp's first row in the tile
  fence_proxy_async_smem();
  __syncwarp();
  if ((r & 31) == 0 && tile_row0 + warp_row < n_rows) {
    for (int c = 0; c < (kCols + 63) / 64 && x0 + c * 64 < d_cols; ++c)
      tma_store_4d(tm, s_tile + c * kChunkBytes + warp_row * 128, x0 + c * 64,
                   tile_row0 + warp_row, h_idx, b_idx);
    bulk_commit_group();
    bulk_wait_group_read0();
  }
  __syncwarp();
}

template <int kCols, bool kF16>
__device__ __noinline__ void store_rows_tma(const CUtensorMap *tm, uint32_t tacc,
                                            uint32_t s_tile, int r, int tile_row0, int x0,
                                            float sc, bool any, int d_cols, int n_rows,
                                            int h_idx, int b_idx) {
  store_rows_tma_inl<kCols, kF16>(tm, tacc, s_tile, r, tile_row0, x0, sc, any, d_cols, n_rows,
                                  h_idx, b_idx);
}

}  // namespace fa
