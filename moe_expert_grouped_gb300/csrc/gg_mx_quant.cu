// gg_mx_quant.cu — MXFP8 quantisers of the expert layer: the permuted
// activation rows (the A operand of FC1 and of the first input-gradient GEMM)
// and the four weight operands, quantised once from the frozen BF16 weights.
// Format and scale-tile layouts: gg_mx.cuh.

#include <cuda_runtime.h>

#include "gg_internal.h"
#include "gg_launch.cuh"
#include "gg_mx.cuh"
#include "gg_ptx.cuh"

namespace gg {
namespace {

__global__ void __launch_bounds__(1024)
tile_prefix_kernel(const int32_t* __restrict__ offsets, int E, int32_t* __restrict__ tb) {
  __shared__ int warp_sums[32];
  grid_dependents_launch();  // the row quantiser waits for this grid's results
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

// One warp per token: the token's row is read once and each 32-element
// block is quantised once (once per pair when the pairs scale it by their
// probability) and written to the permuted row of every pair of the token,
// its scale byte into the 128-row tile of the expert whose rows contain it.
// Lane j < k first resolves pair j's row, its expert (binary search of the
// offsets, staged in shared memory with the scale-tile prefix once per
// block) and its scale position. The row moves in passes of 256 16-byte
// chunks: lane l holds chunks l + 32 i (i < 8), so every load and store
// instruction covers one contiguous stretch of the row, and a block's four
// chunks sit in four neighbouring lanes, which share its maximum. After
// their tokens the warps give code 0 to every scale cell no pair writes
// (units of 32 rows of a scale tile: rows past an expert's end in its last
// tile, padding rows, and the tiles past the last expert's), so the scale
// buffer needs no clearing pass. Launched behind the tile prefix kernel, it
// waits for that kernel's results before reading them.
template <bool kScaled>  // prob != nullptr: each pair's copy is scaled by its probability
__global__ void __launch_bounds__(256)
quantize_scatter_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ row_of_slot,
                        const int32_t* __restrict__ slot_of_row, bool has_padding,
                        const float* __restrict__ prob,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ tb,
                        int T, int k, int K, int E, int R_cap, int sf_tiles_cap,
                        uint8_t* __restrict__ Q, uint8_t* __restrict__ S, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int vec = K / 8;  // 16-byte chunks of a source row; K % 128 == 0
  const int KG = K / mx::kKStep;
  const long long tile_bytes = static_cast<long long>(KG) * mx::kSfaBytes;
  // offsets and tiles_before in shared memory: the searches below would
  // otherwise chain seven global loads per token on the way to its stores
  extern __shared__ int s_tab[];  // [E + 1] offsets, then [E + 1] tiles_before
  int* s_off = s_tab;
  int* s_tb = s_tab + E + 1;
  grid_dependency_wait();  // tiles_before
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_off[i] = offsets[i];
    s_tb[i] = tb[i];
  }
  __syncthreads();
  for (long long t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    long long my_sf = 0;  // byte of block 0 of this pair's row in S
    float my_p = 1.0f;
    if (lane < k) {
      const int row = row_of_slot[t * k + lane];
      int e = 0, hi = E;  // the expert whose rows contain `row`: offsets[e] <= row
      while (hi - e > 1) {
        const int mid = (e + hi) >> 1;
        if (s_off[mid] <= row)
          e = mid;
        else
          hi = mid;
      }
      const int local = row - s_off[e];
      const long long tile = static_cast<long long>(s_tb[e]) + (local >> 7);
      if (row >= 0 && row < R_cap && local >= 0 && row < s_off[e + 1] && tile < sf_tiles_cap) {
        my_row = row;
        my_sf = tile * tile_bytes + mx::sf_byte(local & 127, 0);
      } else if (row != -1) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
      }
      if (kScaled) my_p = prob[t * k + lane];
    }
    const uint4* sp = src + t * vec;
    for (int c0 = 0; c0 < vec; c0 += 256) {
      // chunk c = c0 + lane + 32 i: elements 8c..8c+7, in block c / 4
      uint4 raw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        raw[i] = c < vec ? __ldg(sp + c) : make_uint4(0u, 0u, 0u, 0u);
      }
      uint2 q[8];
      uint32_t sw[8];  // lanes 0 and 16: the scale bytes of the 4 blocks of their 16 chunks
      const auto quantize = [&](float pj) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t code = mx::quantize8x4<kScaled>(raw[i], pj, q[i]);
          const int src0 = lane & 16;
          const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, code, src0 + 4);
          const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, code, src0 + 8);
          const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, code, src0 + 12);
          sw[i] = code | (b1 << 8) | (b2 << 16) | (b3 << 24);
        }
      };
      if (!kScaled) quantize(1.0f);
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xFFFFFFFFu, my_row, j);
        const long long sfo = __shfl_sync(0xFFFFFFFFu, my_sf, j);
        const float pj = __shfl_sync(0xFFFFFFFFu, my_p, j);
        if (row < 0) continue;  // the same for the whole warp
        if (kScaled) quantize(pj);
        uint2* d = reinterpret_cast<uint2*>(Q + static_cast<long long>(row) * K);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < vec) __stcs(d + c, q[i]);
        }
        // the scale bytes of k-step c / 16 (four blocks) as one 32-bit cell
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          if ((lane & 15) == 0 && c < vec)
            *reinterpret_cast<uint32_t*>(S + sfo + static_cast<long long>(c / 16) * mx::kSfaBytes) =
                sw[i];
        }
      }
    }
  }
  // scale cells no pair writes: unit u = (tile u / 4, rows 32 (u % 4) .. +31),
  // unit u to warp (T + u) mod nwarps, so the warps without a token go first
  const long long n_units = static_cast<long long>(sf_tiles_cap) * (mx::kRowTile / 32);
  const int used_tiles = s_tb[E];
  for (long long u = ((warp0 - T) % nwarps + nwarps) % nwarps; u < n_units; u += nwarps) {
    const int tile = static_cast<int>(u >> 2);
    const int r = static_cast<int>(u & 3) * 32 + lane;  // row in the tile
    bool zero = true;
    if (tile < used_tiles) {
      int e = 0, hi = E;  // the expert owning the tile: s_tb[e] <= tile < s_tb[e + 1]
      while (hi - e > 1) {
        const int mid = (e + hi) >> 1;
        if (s_tb[mid] <= tile)
          e = mid;
        else
          hi = mid;
      }
      const int local = (tile - s_tb[e]) * mx::kRowTile + r;
      const long long row = static_cast<long long>(s_off[e]) + local;
      zero = local >= s_off[e + 1] - s_off[e] ||
             (has_padding && (row >= R_cap || slot_of_row[row] < 0));
    }
    if (zero) {
      uint8_t* cell = S + static_cast<long long>(tile) * tile_bytes + mx::sf_byte(r, 0);
      for (int m = 0; m < KG; ++m)
        *reinterpret_cast<uint32_t*>(cell + static_cast<long long>(m) * mx::kSfaBytes) = 0u;
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
      if (gated_F > 0) {  // FC1: gate rows in columns 0..127 of a tile, up rows in 128..255
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
                                    const int32_t* row_of_slot, const int32_t* slot_of_row,
                                    const int32_t* offsets, const int32_t* tiles_before, int E,
                                    int R_cap, bool has_padding, int sf_tiles_cap,
                                    const float* prob, uint8_t* Q, uint8_t* S, int32_t* status,
                                    int sm_count, cudaStream_t stream) {
  if (T < 0 || sf_tiles_cap <= 0) return cudaSuccess;
  // one token per warp, then one warp per 32-row unit of the scale tiles: the
  // blocks, far more than fit at once, start as earlier ones finish, which
  // balances the SMs to within one block
  const long long warps =
      static_cast<long long>(T) + static_cast<long long>(sf_tiles_cap) * (mx::kRowTile / 32);
  long long blocks = (warps + 7) / 8;  // 8 warps per block
  const long long cap = static_cast<long long>(sm_count) * 1024;
  if (blocks > cap) blocks = cap;
  // E <= kMaxExperts: at most 8 KB of staged tables
  const size_t tab_bytes = sizeof(int) * 2 * (static_cast<size_t>(E) + 1);
  const dim3 grid(static_cast<unsigned>(blocks)), block(256);
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  // behind the tile prefix kernel: started early, waits for tiles_before
  cudaError_t e =
      prob != nullptr
          ? launch_early(quantize_scatter_kernel<true>, grid, block, tab_bytes, stream, s4,
                         row_of_slot, slot_of_row, has_padding, prob, offsets, tiles_before, T,
                         k, K, E, R_cap, sf_tiles_cap, Q, S, status)
          : launch_early(quantize_scatter_kernel<false>, grid, block, tab_bytes, stream, s4,
                         row_of_slot, slot_of_row, has_padding, prob, offsets, tiles_before, T,
                         k, K, E, R_cap, sf_tiles_cap, Q, S, status);
  if (e != cudaSuccess) return e;
  count_launch();
  if (has_padding)  // E4M3 zeros on the padding rows (K bytes = K/16 vectors)
    return launch_zero_pad_rows(slot_of_row, offsets, E, R_cap, K / 16, Q, sm_count, stream);
  return cudaSuccess;
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
