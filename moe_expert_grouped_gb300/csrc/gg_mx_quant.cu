// gg_mx_quant.cu — MXFP8 quantisers of the expert layer: the permuted
// activation rows (the A operand of FC1 and of the first input-gradient GEMM)
// and the four weight operands, quantised once from the frozen BF16 weights.
// Format and scale-tile layouts: gg_mx.cuh.

#include <cuda_runtime.h>

#include "gg_internal.h"
#include "gg_mx.cuh"
#include "gg_ptx.cuh"

namespace gg {
namespace {

__global__ void __launch_bounds__(1024)
tile_prefix_kernel(const int32_t* __restrict__ offsets, int E, int32_t* __restrict__ tb) {
  __shared__ int warp_sums[32];
  const int t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  int v = 0;
  if (t < E) {
    const int n = offsets[t + 1] - offsets[t];
    v = n > 0 ? (n + mx::kRowTile - 1) / mx::kRowTile : 0;
  }
  int incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, s, d);
      if (lane >= d) s += n;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const int excl = incl - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (t < E) tb[t] = excl;
  if (t == E - 1) tb[E] = excl + v;
}

__device__ __forceinline__ void unpack_bf16x8(uint4 w, float* v) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

// One warp per row of every expert's 128-row tiles; lane b handles the
// 32-element blocks b, b + 32, ... of the row (64 contiguous source bytes in,
// 32 bytes out per block).
__global__ void __launch_bounds__(256)
quantize_rows_kernel(const gg_bf16* __restrict__ src, int T, int K, int k,
                     const int32_t* __restrict__ slot_of_row, const int32_t* __restrict__ offsets,
                     const int32_t* __restrict__ tb, int E, int R_cap, int sf_tiles_cap,
                     const float* __restrict__ prob_of_row, uint8_t* __restrict__ Q,
                     uint8_t* __restrict__ S, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  int total_tiles = tb[E];
  if (total_tiles > sf_tiles_cap) {
    if (warp_id == 0 && lane == 0) set_status(status, GG_ERR_DEVICE_BAD_OFFSETS);
    total_tiles = sf_tiles_cap;
  }
  const int KG = K / mx::kKStep;
  const int nblk = K / mx::kBlock;
  const long long pairs = static_cast<long long>(T) * k;
  for (long long w = warp_id; w < static_cast<long long>(total_tiles) * mx::kRowTile;
       w += n_warps) {
    const int tile = static_cast<int>(w / mx::kRowTile);
    const int r = static_cast<int>(w % mx::kRowTile);
    int lo = 0, hi = E;  // tb[lo] <= tile < tb[lo + 1]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tb[mid] <= tile)
        lo = mid;
      else
        hi = mid;
    }
    const int e = lo;
    const long long grow =
        static_cast<long long>(offsets[e]) + static_cast<long long>(tile - tb[e]) * mx::kRowTile + r;
    const bool in_expert = grow < offsets[e + 1] && grow < R_cap;
    long long src_row = -1;
    float p = 1.0f;
    if (in_expert) {
      const int slot = slot_of_row[grow];
      if (slot >= pairs) {
        if (lane == 0) set_status(status, GG_ERR_DEVICE_BAD_ROW);
      } else if (slot >= 0) {
        src_row = slot / k;
      }
      if (prob_of_row != nullptr) p = prob_of_row[grow];
    }
    const uint4* srow = reinterpret_cast<const uint4*>(src + (src_row >= 0 ? src_row : 0) * K);
    for (int b = lane; b < nblk; b += 32) {
      float v[32];
      if (src_row >= 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) unpack_bf16x8(__ldg(srow + 4 * b + j), v + 8 * j);
        if (prob_of_row != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = round_bf16(v[i] * p);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      }
      uint32_t q[8];
      const uint32_t code = mx::quantize32(v, q);
      if (in_expert) {
        uint4* d = reinterpret_cast<uint4*>(Q + grow * K + b * mx::kBlock);
        d[0] = make_uint4(q[0], q[1], q[2], q[3]);
        d[1] = make_uint4(q[4], q[5], q[6], q[7]);
      }
      S[(static_cast<long long>(tile) * KG + (b >> 2)) * mx::kSfaBytes + mx::sf_byte(r, b & 3)] =
          static_cast<uint8_t>(in_expert ? code : 0u);
    }
  }
}

// A 32 x 32 tile of one expert's weight per block: loaded coalesced in the
// source orientation, read back row by row of the operand; one thread per
// operand row quantises its 32-element block.
__global__ void __launch_bounds__(256)
prepare_weight_kernel(const gg_bf16* __restrict__ W, int N, int K, int transpose, int gated_F,
                      int NT, uint8_t* __restrict__ Wq, uint8_t* __restrict__ S) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32;
  const int n0 = blockIdx.y * 32;
  const long long e = blockIdx.z;
  const unsigned short* Wu = reinterpret_cast<const unsigned short*>(W);
  for (int i = threadIdx.x; i < 32 * 32; i += blockDim.x) {
    const int a = i >> 5, b = i & 31;
    if (!transpose) {  // W [E][N][K]: element (n0 + a, k0 + b)
      const int n = n0 + a;
      tile[a][b] = n < N ? __uint_as_float(static_cast<uint32_t>(Wu[(e * N + n) * K + k0 + b])
                                           << 16)
                         : 0.0f;
    } else {  // W [E][K][N]: element (n0 + b, k0 + a)
      const int n = n0 + b;
      tile[b][a] = n < N ? __uint_as_float(static_cast<uint32_t>(Wu[(e * K + k0 + a) * N + n])
                                           << 16)
                         : 0.0f;
    }
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int n = n0 + threadIdx.x;
    if (n < N) {
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = tile[threadIdx.x][j];
      uint32_t q[8];
      const uint32_t code = mx::quantize32(v, q);
      uint4* d = reinterpret_cast<uint4*>(Wq + (e * N + n) * K + k0);
      d[0] = make_uint4(q[0], q[1], q[2], q[3]);
      d[1] = make_uint4(q[4], q[5], q[6], q[7]);
      int nt, col;
      if (gated_F > 0) {  // FC1: gate rows in columns 0..95 of a tile, up rows in 96..191
        const bool up = n >= gated_F;
        const int j = up ? n - gated_F : n;
        nt = j / mx::kTileNHalf;
        col = j % mx::kTileNHalf + (up ? mx::kTileNHalf : 0);
      } else {
        nt = n / mx::kTileN;
        col = n % mx::kTileN;
      }
      const int KG = K / mx::kKStep;
      S[((e * NT + nt) * KG + k0 / mx::kKStep) * mx::kSfbBytes +
        mx::sfb_byte(col, (k0 / mx::kBlock) & 3)] = static_cast<uint8_t>(code);
    }
  }
}

}  // namespace

cudaError_t launch_mx_tile_prefix(const int32_t* offsets, int E, int32_t* tiles_before,
                                  cudaStream_t stream) {
  if (E <= 0 || E > 1024) return cudaErrorInvalidValue;
  tile_prefix_kernel<<<1, 1024, 0, stream>>>(offsets, E, tiles_before);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mx_quantize_rows(const gg_bf16* src, int T, int K, int k,
                                    const int32_t* slot_of_row, const int32_t* offsets,
                                    const int32_t* tiles_before, int E, int R_cap,
                                    int sf_tiles_cap, const float* prob_of_row, uint8_t* Q,
                                    uint8_t* S, int32_t* status, int sm_count,
                                    cudaStream_t stream) {
  if (sf_tiles_cap <= 0) return cudaSuccess;
  const long long rows = static_cast<long long>(sf_tiles_cap) * mx::kRowTile;
  long long blocks = (rows + 7) / 8;  // 8 warps per block
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  quantize_rows_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
      src, T, K, k, slot_of_row, offsets, tiles_before, E, R_cap, sf_tiles_cap, prob_of_row, Q, S,
      status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_mx_prepare_weight(const gg_bf16* W, int E, int N, int K, bool transpose,
                                     int gated_F, int NT, uint8_t* Wq, uint8_t* S,
                                     cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(K / 32), static_cast<unsigned>((N + 31) / 32),
                  static_cast<unsigned>(E));
  prepare_weight_kernel<<<grid, 256, 0, stream>>>(W, N, K, transpose ? 1 : 0, gated_F, NT, Wq, S);
  count_launch();
  return cudaGetLastError();
}

}  // namespace gg
