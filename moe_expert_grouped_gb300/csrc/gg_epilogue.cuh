// gg_epilogue.cuh — device helpers shared by the grouped GEMM epilogues
// (BF16 and MXFP8): work-item decoding and the warp-staged row-contiguous
// stores and loads of 32-row chunks.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "gg_ptx.cuh"

namespace gg {
namespace {

// Work item `tile` -> (expert e, row-block pair mt, column block nt), with
// tb[e] the first work item of expert e (tb[E] = total) and NT column blocks
// per row-block pair.
__device__ __forceinline__ void decode_tile(int tile, const int* tb, int E, int NT, int& e,
                                            int& mt, int& nt) {
  int lo = 0, hi = E;  // tb[lo] <= tile < tb[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tb[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  e = lo;
  const int local = tile - tb[lo];
  mt = local / NT;
  nt = local - mt * NT;
}

__device__ __forceinline__ void pack_bf16x32(const float (&v)[32], float scale, uint4 (&w)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[i].x = pack_bf16x2(v[8 * i + 0] * scale, v[8 * i + 1] * scale);
    w[i].y = pack_bf16x2(v[8 * i + 2] * scale, v[8 * i + 3] * scale);
    w[i].z = pack_bf16x2(v[8 * i + 4] * scale, v[8 * i + 5] * scale);
    w[i].w = pack_bf16x2(v[8 * i + 6] * scale, v[8 * i + 7] * scale);
  }
}

// 16-byte slot of column group c (0..3) of row r (0..31) in a warp's staging
// buffer; the XOR spreads every 8-lane shared-memory phase over all banks.
__device__ __forceinline__ int stage_slot(int r, int c) { return r * 4 + (c ^ ((r >> 1) & 3)); }

// Warp-collective store of a 32-row x 32-column BF16 chunk. Lane i holds row
// i in w[]; row r of the chunk starts at row0 + r * ld (the warp's 32 rows
// are consecutive) and only rows r < nvalid are written. Through the staging
// buffer four lanes write each 64-byte row segment, so every store
// instruction writes 8 whole row segments instead of 32 scattered 16-byte
// pieces.
__device__ __forceinline__ void store_chunk(uint4* stg, const uint4 (&w)[4], gg_bf16* row0,
                                            long long ld, int nvalid) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 4; ++c) stg[stage_slot(lane, c)] = w[c];
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 8 * j + (lane >> 2);
    const int c = lane & 3;
    const uint4 v = stg[stage_slot(r, c)];
    if (r < nvalid) reinterpret_cast<uint4*>(row0 + r * ld)[c] = v;
  }
  __syncwarp();
}

// Warp-collective coalesced fetch of a 32-row x 32-column BF16 chunk (rows
// row0 + r * ld): lane L loads column group L%4 of rows 8j + L/4 (raw
// layout); rows r >= nvalid read as zero. transpose_chunk() then hands each
// lane its own row.
__device__ __forceinline__ void load_chunk_raw(uint4 (&raw)[4], const gg_bf16* row0, long long ld,
                                               int nvalid) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = 8 * j + (lane >> 2);
    raw[j] = r < nvalid ? __ldg(reinterpret_cast<const uint4*>(row0 + r * ld) + (lane & 3))
                        : make_uint4(0u, 0u, 0u, 0u);
  }
}

__device__ __forceinline__ void transpose_chunk(uint4* stg, const uint4 (&raw)[4], uint4 (&w)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 4; ++j) stg[stage_slot(8 * j + (lane >> 2), lane & 3)] = raw[j];
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) w[c] = stg[stage_slot(lane, c)];
  __syncwarp();
}

}  // namespace
}  // namespace gg
