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

// One warp per token: the token's row is read once and each 32-element
// block is quantised once (once per pair when the pairs scale it by their
// probability) and written to the permuted row of every pair of the token,
// its scale byte into the 128-row tile of the expert whose rows contain it.
// Lane b0 + l owns block b0 + l; lane j < k first resolves pair j's row, its
// expert (binary search of the offsets, staged in shared memory with the
// scale-tile prefix once per block) and its scale position.
template <bool kScaled>  // prob != nullptr: each pair's copy is scaled by its probability
__global__ void __launch_bounds__(256)
quantize_scatter_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ row_of_slot,
                        const float* __restrict__ prob,
                        const int32_t* __restrict__ offsets, const int32_t* __restrict__ tb,
                        int T, int k, int K, int E, int R_cap, int sf_tiles_cap,
                        uint8_t* __restrict__ Q, uint8_t* __restrict__ S, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int nblk = K / mx::kBlock;
  const long long tile_bytes = static_cast<long long>(K / mx::kKStep) * mx::kSfaBytes;
  // offsets and tiles_before in shared memory: the searches below would
  // otherwise chain seven global loads per token on the way to its stores
  extern __shared__ int s_tab[];  // [E + 1] offsets, then [E + 1] tiles_before
  int* s_off = s_tab;
  int* s_tb = s_tab + E + 1;
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
    const uint4* sp = src + t * (K / 8);
    // two blocks per lane and pass: their eight 16-byte loads are in flight together
    for (int b0 = 0; b0 < nblk; b0 += 64) {
      uint4 raw[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = b0 + 32 * h + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          raw[h][j] = b < nblk ? __ldg(sp + 4 * b + j) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int b = b0 + 32 * h + lane;
        const bool live = b < nblk;
        float v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) unpack_bf16x8(raw[h][j], v + 8 * j);
        const long long sf_b = (b >> 2) * static_cast<long long>(mx::kSfaBytes) + (b & 3);
        uint32_t q[8];
        uint32_t code = kScaled ? 0u : mx::quantize32(v, q);
        for (int j = 0; j < k; ++j) {
          const int row = __shfl_sync(0xFFFFFFFFu, my_row, j);
          const long long sfo = __shfl_sync(0xFFFFFFFFu, my_sf, j);
          const float pj = __shfl_sync(0xFFFFFFFFu, my_p, j);
          if (row < 0) continue;
          if (kScaled) {
            float w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = round_bf16(v[i] * pj);
            code = mx::quantize32(w, q);
          }
          if (live) {
            uint4* d =
                reinterpret_cast<uint4*>(Q + static_cast<long long>(row) * K + b * mx::kBlock);
            __stcs(d, make_uint4(q[0], q[1], q[2], q[3]));
            __stcs(d + 1, make_uint4(q[4], q[5], q[6], q[7]));
            S[sfo + sf_b] = static_cast<uint8_t>(code);
          }
        }
      }
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
  // code 0 wherever no pair lands: rows past an expert's end, padding rows
  cudaError_t e = cudaMemsetAsync(
      S, 0, static_cast<size_t>(sf_tiles_cap) * (K / mx::kKStep) * mx::kSfaBytes, stream);
  if (e != cudaSuccess || T <= 0) return e;
  long long blocks = (static_cast<long long>(T) + 7) / 8;  // 8 warps per block
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  // E <= kMaxExperts: at most 8 KB of staged tables
  const size_t tab_bytes = sizeof(int) * 2 * (static_cast<size_t>(E) + 1);
  if (prob != nullptr)
    quantize_scatter_kernel<true><<<static_cast<int>(blocks), 256, tab_bytes, stream>>>(
        reinterpret_cast<const uint4*>(src), row_of_slot, prob, offsets, tiles_before, T, k, K,
        E, R_cap, sf_tiles_cap, Q, S, status);
  else
    quantize_scatter_kernel<false><<<static_cast<int>(blocks), 256, tab_bytes, stream>>>(
        reinterpret_cast<const uint4*>(src), row_of_slot, prob, offsets, tiles_before, T, k, K,
        E, R_cap, sf_tiles_cap, Q, S, status);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
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
