// gg_permute.cu — memory-bound kernels of the expert layer: the routed-token
// permute (stable counting sort of (token, slot) pairs by expert plus the row
// gather), the gather of a token-major gradient into permuted order, and the
// probability-weighted combine. Sources: "perf(moe): add frozen grouped GEMM
// for adapter training" (AlignmentResearch/Megatron-LM PR #3), "B200
// throughput evidence" (tokens grouped by expert after all-to-all dispatch);
// NVIDIA/Megatron-LM PR #7333 "Summary" (256-row expert padding); "[Main]
// Support paged stash with device-initiated GroupedLinear" (NVIDIA/Megatron-LM
// PR #6828), "What does this PR do?" (probability boundary).
//
// Determinism: every index is computed by counting, never by atomics whose
// order matters, so row maps are bit-exact and run-to-run identical. The
// combine sums a token's k slots in slot order in fp32 with one rounding.

#include <cuda_runtime.h>

#include <atomic>

#include "gg_internal.h"
#include "gg_launch.cuh"
#include "gg_ptx.cuh"

namespace gg {
namespace {

constexpr int kWarps = kPermuteBlockThreads / 32;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Expert of pair p, or -1 for p >= R and for an id outside [0, E) (reported
// when status is not null).
__device__ __forceinline__ int pair_expert(const int32_t* __restrict__ idx, long long p,
                                           long long R, int E, int32_t* status) {
  if (p >= R) return -1;
  const int e = idx[p];
  if (e < 0 || e >= E) {
    if (status != nullptr) set_status(status, GG_ERR_DEVICE_BAD_EXPERT_ID);
    return -1;
  }
  return e;
}

// Block b counts the experts of pairs [b ppb, (b + 1) ppb) into
// block_hist[b][E]. It also marks every row as padding (slot -1, probability
// 0); the scatter kernel fills in the routed rows.
__global__ void __launch_bounds__(kPermuteBlockThreads)
permute_count_kernel(const int32_t* __restrict__ idx, long long R, int E, long long ppb,
                     int32_t* __restrict__ block_hist, int32_t* status,
                     int32_t* __restrict__ slot_of_row, float* __restrict__ prob_of_row,
                     long long R_cap) {
  grid_dependents_launch();  // the scatter kernel waits for this grid's results
  for (long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < R_cap;
       r += static_cast<long long>(gridDim.x) * blockDim.x) {
    slot_of_row[r] = -1;
    prob_of_row[r] = 0.0f;
  }
  extern __shared__ int hist[];  // [E]
  for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long first = static_cast<long long>(blockIdx.x) * ppb;
  const long long last = min(R, first + ppb);
#pragma unroll 1
  for (long long p0 = first + 32LL * warp; p0 < last; p0 += kPermuteBlockThreads) {
    const int e = pair_expert(idx, p0 + lane, last, E, status);
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0 && (peers & lanemask_lt()) == 0) atomicAdd(&hist[e], __popc(peers));
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    block_hist[static_cast<long long>(blockIdx.x) * E + e] = hist[e];
}

// Block b of the scatter (nb = number of count blocks; one block when nb = 0):
//  (1) from all nb histogram rows, every expert's total count and the count in
//      the blocks before b (each of the 1024 / E threads of an expert sums a
//      range of rows with its loads in flight together);
//  (2) offsets = exclusive prefix of the totals padded to multiples of P
//      (written by block 0);
//  (3) the per-warp histograms of its own pairs (warp w owns the contiguous
//      pairs [b ppb + w ppb / 32, +ppb / 32), 32 at a time), turned into
//      running row bases: expert e's rows for warp w of block b start at
//      offsets[e] + (count of e before b) + (count of e in warps < w);
//  (4) stable rows: each warp walks its pairs in order, a pair's row is its
//      warp base plus the number of earlier lanes of the step with the same
//      expert. No order-dependent atomics anywhere: the maps are bit-exact.
__global__ void __launch_bounds__(kPermuteBlockThreads)
permute_scatter_kernel(const int32_t* __restrict__ idx, const float* __restrict__ prob,
                       long long R, int E, int P, long long ppb, int nb,
                       const int32_t* __restrict__ block_hist, int32_t* __restrict__ offsets,
                       int32_t* __restrict__ row_of_slot, int32_t* __restrict__ slot_of_row,
                       float* __restrict__ prob_of_row) {
  extern __shared__ int sm[];
  int* wb = sm;                          // [kWarps][E]: warp counts, then warp row bases
  int* part_all = wb + kWarps * E;       // [kPermuteBlockThreads]
  int* part_below = part_all + kPermuteBlockThreads;
  int* base_e = part_below + kPermuteBlockThreads;  // [E]: offsets[e] + count before b
  __shared__ int warp_tot[kWarps];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int b = blockIdx.x;
  grid_dependents_launch();  // the row copy waits for this grid's results
  // zero the warp histograms while the count kernel finishes
  for (int i = t; i < kWarps * E; i += kPermuteBlockThreads) wb[i] = 0;
  grid_dependency_wait();  // block_hist, and slot_of_row marked as padding

  // (1) totals and counts before this block
  const int parts = max(1, kPermuteBlockThreads / E);
  {
    const int e = t % E, part = t / E;
    int s_all = 0, s_below = 0;
    if (part < parts && t < parts * E) {
      const int b0 = static_cast<int>((static_cast<long long>(nb) * part) / parts);
      const int b1 = static_cast<int>((static_cast<long long>(nb) * (part + 1)) / parts);
      constexpr int kChunk = 8;
      for (int r0 = b0; r0 < b1; r0 += kChunk) {
        int v[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j)
          v[j] = r0 + j < b1 ? block_hist[static_cast<long long>(r0 + j) * E + e] : 0;
#pragma unroll
        for (int j = 0; j < kChunk; ++j) {
          s_all += v[j];
          if (r0 + j < b) s_below += v[j];
        }
      }
    }
    part_all[t] = s_all;
    part_below[t] = s_below;
  }
  __syncthreads();

  // (2) padded exclusive prefix over experts, E <= 1024 = one expert per thread
  int total = 0, below = 0;
  if (t < E) {
    for (int q = 0; q < parts; ++q) {
      total += part_all[q * E + t];
      below += part_below[q * E + t];
    }
  }
  const int padded = t < E ? (total + P - 1) / P * P : 0;
  int incl = padded;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
    if (lane >= d) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xFFFFFFFFu, w, d);
      if (lane >= d) w += n;
    }
    warp_tot[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int excl = incl - padded + (warp > 0 ? warp_tot[warp - 1] : 0);
  if (t < E) {
    base_e[t] = excl + below;
    if (b == 0) {
      offsets[t] = excl;
      if (t == E - 1) offsets[E] = excl + padded;
    }
  }

  // (3) per-warp histograms of this block's pairs
  const long long first = static_cast<long long>(b) * ppb;
  const long long last = min(R, first + ppb);
  const long long ppw = ppb / kWarps;
  const long long wfirst = first + ppw * warp;
  const long long wlast = min(last, wfirst + ppw);
  int* hw = wb + warp * E;
#pragma unroll 1
  for (long long p0 = wfirst; p0 < wlast; p0 += 32) {
    const int e = pair_expert(idx, p0 + lane, wlast, E, nullptr);
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    if (e >= 0 && (peers & lanemask_lt()) == 0) hw[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = t; e < E; e += kPermuteBlockThreads) {
    int run = base_e[e];
#pragma unroll 4
    for (int w = 0; w < kWarps; ++w) {
      const int c = wb[w * E + e];
      wb[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();

  // (4) stable rows
#pragma unroll 1
  for (long long p0 = wfirst; p0 < wlast; p0 += 32) {
    const long long p = p0 + lane;
    const int e = pair_expert(idx, p, wlast, E, nullptr);
    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
    int row = -1;
    if (e >= 0) row = hw[e] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (e >= 0 && (peers & lanemask_lt()) == 0) hw[e] += __popc(peers);
    __syncwarp();
    if (p < wlast) {
      row_of_slot[p] = row;
      if (row >= 0) {
        slot_of_row[row] = static_cast<int32_t>(p);
        prob_of_row[row] = prob[p];
      }
    }
  }
}

// Zero the padding rows (slot -1) below offsets[E]. The work is cut into
// units of one 32-row group by one column slice of up to 64 16-byte vectors;
// a unit is a ballot over the group's slots, then the slice cleared on the
// group's padding rows. Padding rows come in runs at the ends of the experts'
// segments, so the heavy units are neighbours: warp w of the nw (nw a
// multiple of 8, the warps of 256-thread blocks) takes the units
// u = (w % 8) * (nw / 8) + w / 8 + i * nw, i = 0, 1, ..., which puts
// neighbouring units in different blocks and so spreads a run over the SMs.
__device__ __forceinline__ void zero_pad_rows(const int32_t* __restrict__ slot_of_row,
                                              const int32_t* __restrict__ offsets, int E,
                                              int R_cap, int vec_per_row,
                                              uint4* __restrict__ dst, long long w,
                                              long long nw) {
  constexpr int kSlice = 64;
  const int lane = threadIdx.x & 31;
  // offsets may come from the caller: never past the buffer's R_cap rows
  const long long n_rows = min(static_cast<long long>(offsets[E]), static_cast<long long>(R_cap));
  const long long n_slices = (vec_per_row + kSlice - 1) / kSlice;
  const long long n_units = (n_rows + 31) / 32 * n_slices;
  const long long first = nw % 8 == 0 ? (w % 8) * (nw / 8) + w / 8 : w;
  for (long long u = first; u < n_units; u += nw) {
    const long long g = u / n_slices;
    const int c_lo = static_cast<int>(u - g * n_slices) * kSlice;
    const int c_hi = min(vec_per_row, c_lo + kSlice);
    const long long base = g * 32;
    const long long r = base + lane;
    const bool pad = r < n_rows && slot_of_row[r] < 0;
    uint32_t mask = __ballot_sync(0xFFFFFFFFu, pad);
    while (mask != 0) {
      const int b = __ffs(mask) - 1;
      mask &= mask - 1;
      uint4* d = dst + (base + b) * vec_per_row;
      for (int c = c_lo + lane; c < c_hi; c += 32) __stcs(d + c, make_uint4(0u, 0u, 0u, 0u));
    }
  }
}

// dst[row_of_slot[t*k+j]] = src[t] for every pair (t, j) with a row: one warp
// per token reads the token's row once and writes its k copies (reading the
// source in order and writing whole 16-byte-vector rows runs at copy speed;
// the destination-ordered form re-reads source rows through L2 in random
// order). Stores are streaming: the permuted buffer is far larger than L2.
// With slot_of_row given, the same launch then zeroes the padding rows
// below offsets[E] (each warp after its tokens, so the copy and the zeroing
// overlap instead of running back to back).
__global__ void __launch_bounds__(256)
scatter_rows_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ row_of_slot,
                    int T, int k, int vec_per_row, int R_cap, uint4* __restrict__ dst,
                    int32_t* status, const int32_t* __restrict__ pad_slot_of_row,
                    const int32_t* __restrict__ offsets, int E) {
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  grid_dependency_wait();  // the row maps, when launched behind their writer
  for (long long t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    if (lane < k) {
      my_row = row_of_slot[t * k + lane];
      if (my_row < -1 || my_row >= R_cap) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
        my_row = -1;
      }
    }
    const uint4* sp = src + t * vec_per_row;
    for (int c0 = 0; c0 < vec_per_row; c0 += 256) {
      uint4 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        a[i] = c < vec_per_row ? __ldg(sp + c) : make_uint4(0u, 0u, 0u, 0u);
      }
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xFFFFFFFFu, my_row, j & 31);
        if (row < 0) continue;
        uint4* d = dst + static_cast<long long>(row) * vec_per_row;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < vec_per_row) __stcs(d + c, a[i]);
        }
      }
    }
  }
  if (pad_slot_of_row != nullptr)
    zero_pad_rows(pad_slot_of_row, offsets, E, R_cap, vec_per_row, dst, warp0, nwarps);
}

// scatter_rows_kernel with the pre-FC1 probability multiply: the copy of
// token t for pair (t, j) is bf16(prob[t*k+j] * src[t]), the product in fp32.
__global__ void __launch_bounds__(256)
scatter_rows_scaled_kernel(const uint4* __restrict__ src, const int32_t* __restrict__ row_of_slot,
                           const float* __restrict__ prob, int T, int k, int vec_per_row,
                           int R_cap, uint4* __restrict__ dst, int32_t* status,
                           const int32_t* __restrict__ pad_slot_of_row,
                           const int32_t* __restrict__ offsets, int E) {
  const int lane = threadIdx.x & 31;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  grid_dependency_wait();  // the row maps, when launched behind their writer
  for (long long t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    float my_p = 0.0f;
    if (lane < k) {
      my_row = row_of_slot[t * k + lane];
      my_p = prob[t * k + lane];
      if (my_row < -1 || my_row >= R_cap) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
        my_row = -1;
      }
    }
    const uint4* sp = src + t * vec_per_row;
    for (int c0 = 0; c0 < vec_per_row; c0 += 256) {
      uint4 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = c0 + lane + 32 * i;
        a[i] = c < vec_per_row ? __ldg(sp + c) : make_uint4(0u, 0u, 0u, 0u);
      }
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xFFFFFFFFu, my_row, j & 31);
        const float pj = __shfl_sync(0xFFFFFFFFu, my_p, j & 31);
        if (row < 0) continue;
        uint4* d = dst + static_cast<long long>(row) * vec_per_row;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + lane + 32 * i;
          if (c < vec_per_row) {
            const uint32_t w[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
              o[q] = pack_bf16x2(pj * bf16_lo(w[q]), pj * bf16_hi(w[q]));
            __stcs(d + c, make_uint4(o[0], o[1], o[2], o[3]));
          }
        }
      }
    }
  }
  if (pad_slot_of_row != nullptr)
    zero_pad_rows(pad_slot_of_row, offsets, E, R_cap, vec_per_row, dst, warp0, nwarps);
}

// Zero the padding rows (slot -1) below offsets[E] (the standalone form, for
// buffers no row copy writes).
__global__ void __launch_bounds__(256)
zero_pad_rows_kernel(const int32_t* __restrict__ slot_of_row, const int32_t* __restrict__ offsets,
                     int E, int R_cap, int vec_per_row, uint4* __restrict__ dst) {
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  zero_pad_rows(slot_of_row, offsets, E, R_cap, vec_per_row, dst, warp0, nwarps);
}

// out[t] = bf16(sum_j prob[t][j] * Yp[row_of_slot[t*k+j]]), fp32 in slot
// order; prob == nullptr gives the plain sum. One warp per token; per pass a
// lane accumulates two 16-byte column groups over the k slots (streaming
// loads, unrolled so that several slots' loads are in flight).
__global__ void __launch_bounds__(256)
combine_kernel(const uint4* __restrict__ Yp, const int32_t* __restrict__ row_of_slot,
               const float* __restrict__ prob, int T, int k, int vec_per_row, int R_cap,
               uint4* __restrict__ out, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    float my_p = 1.0f;
    if (lane < k) {
      my_row = row_of_slot[static_cast<long long>(t) * k + lane];
      if (prob != nullptr) my_p = prob[static_cast<long long>(t) * k + lane];
      if (my_row < -1 || my_row >= R_cap) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
        my_row = -1;
      }
    }
    // The column loop is warp-uniform so that the shuffles below see every lane.
    for (int c0 = 0; c0 < vec_per_row; c0 += 64) {
      const int ca = c0 + lane, cb = c0 + 32 + lane;
      const bool oka = ca < vec_per_row, okb = cb < vec_per_row;
      float acc[2][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[0][i] = acc[1][i] = 0.0f;
#pragma unroll 8
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xFFFFFFFFu, my_row, j & 31);
        const float pj = __shfl_sync(0xFFFFFFFFu, my_p, j & 31);
        if (row < 0) continue;  // warp-uniform: every lane holds the same row
        const uint4* rp = Yp + static_cast<long long>(row) * vec_per_row;
        const uint4 va = oka ? __ldcs(rp + ca) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 vb = okb ? __ldcs(rp + cb) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
        const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[0][2 * q] = __fmaf_rn(pj, bf16_lo(wa[q]), acc[0][2 * q]);
          acc[0][2 * q + 1] = __fmaf_rn(pj, bf16_hi(wa[q]), acc[0][2 * q + 1]);
          acc[1][2 * q] = __fmaf_rn(pj, bf16_lo(wb[q]), acc[1][2 * q]);
          acc[1][2 * q + 1] = __fmaf_rn(pj, bf16_hi(wb[q]), acc[1][2 * q + 1]);
        }
      }
      uint4* op = out + static_cast<long long>(t) * vec_per_row;
      if (oka)
        __stcs(op + ca, make_uint4(pack_bf16x2(acc[0][0], acc[0][1]), pack_bf16x2(acc[0][2], acc[0][3]),
                                   pack_bf16x2(acc[0][4], acc[0][5]), pack_bf16x2(acc[0][6], acc[0][7])));
      if (okb)
        __stcs(op + cb, make_uint4(pack_bf16x2(acc[1][0], acc[1][1]), pack_bf16x2(acc[1][2], acc[1][3]),
                                   pack_bf16x2(acc[1][4], acc[1][5]), pack_bf16x2(acc[1][6], acc[1][7])));
    }
  }
}

// combine_kernel plus the routing-probability gradient: after the column
// loop, lane j < k adds up the n_rowdot partial sums of its pair's row in fp32
// in ascending order (loading them only then keeps the column loop's
// registers, and so its occupancy, those of the plain combine). A separate
// kernel so that the plain combine keeps its own code.
__global__ void __launch_bounds__(256)
combine_dprob_kernel(const uint4* __restrict__ Yp, const int32_t* __restrict__ row_of_slot,
                     const float* __restrict__ prob, int T, int k, int vec_per_row, int R_cap,
                     uint4* __restrict__ out, const float* __restrict__ rowdot, int n_rowdot,
                     float* __restrict__ dprob, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    float my_p = 1.0f;
    if (lane < k) {
      my_row = row_of_slot[static_cast<long long>(t) * k + lane];
      if (prob != nullptr) my_p = prob[static_cast<long long>(t) * k + lane];
      if (my_row < -1 || my_row >= R_cap) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
        my_row = -1;
      }
    }
    const int rd_stride = (n_rowdot + 7) / 8 * 8;
    // The column loop is warp-uniform so that the shuffles below see every lane.
    for (int c0 = 0; c0 < vec_per_row; c0 += 64) {
      const int ca = c0 + lane, cb = c0 + 32 + lane;
      const bool oka = ca < vec_per_row, okb = cb < vec_per_row;
      float acc[2][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[0][i] = acc[1][i] = 0.0f;
#pragma unroll 8
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xFFFFFFFFu, my_row, j & 31);
        const float pj = __shfl_sync(0xFFFFFFFFu, my_p, j & 31);
        if (row < 0) continue;  // warp-uniform: every lane holds the same row
        const uint4* rp = Yp + static_cast<long long>(row) * vec_per_row;
        const uint4 va = oka ? __ldcs(rp + ca) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 vb = okb ? __ldcs(rp + cb) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
        const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[0][2 * q] = __fmaf_rn(pj, bf16_lo(wa[q]), acc[0][2 * q]);
          acc[0][2 * q + 1] = __fmaf_rn(pj, bf16_hi(wa[q]), acc[0][2 * q + 1]);
          acc[1][2 * q] = __fmaf_rn(pj, bf16_lo(wb[q]), acc[1][2 * q]);
          acc[1][2 * q + 1] = __fmaf_rn(pj, bf16_hi(wb[q]), acc[1][2 * q + 1]);
        }
      }
      uint4* op = out + static_cast<long long>(t) * vec_per_row;
      if (oka)
        __stcs(op + ca, make_uint4(pack_bf16x2(acc[0][0], acc[0][1]), pack_bf16x2(acc[0][2], acc[0][3]),
                                   pack_bf16x2(acc[0][4], acc[0][5]), pack_bf16x2(acc[0][6], acc[0][7])));
      if (okb)
        __stcs(op + cb, make_uint4(pack_bf16x2(acc[1][0], acc[1][1]), pack_bf16x2(acc[1][2], acc[1][3]),
                                   pack_bf16x2(acc[1][4], acc[1][5]), pack_bf16x2(acc[1][6], acc[1][7])));
    }
    if (lane < k) {
      float dp = 0.0f;
      if (my_row >= 0) {
        const float* rd = rowdot + static_cast<long long>(my_row) * rd_stride;
#pragma unroll 8
        for (int b = 0; b < n_rowdot; ++b) dp += __ldg(rd + b);
      }
      dprob[static_cast<long long>(t) * k + lane] = dp;
    }
  }
}

// combine_kernel plus the pre-FC1 probability gradient: with Xp[row] =
// prob * dot_src[t], dprob[t*k+j] = <dot_src[t], Yp[row(t, j)]>. Each lane
// keeps one partial dot per slot over its columns (x chunk loaded once per
// pass), reduced across the warp in a fixed butterfly order at the end;
// kMaxK (8 or 32) bounds k and the partials held in registers.
template <int kMaxK>
__global__ void __launch_bounds__(256)
combine_dot_kernel(const uint4* __restrict__ Yp, const int32_t* __restrict__ row_of_slot,
                   const float* __restrict__ prob, int T, int k, int vec_per_row, int R_cap,
                   uint4* __restrict__ out, const uint4* __restrict__ dot_src,
                   float* __restrict__ dprob, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    float my_p = 1.0f;
    if (lane < k) {
      my_row = row_of_slot[static_cast<long long>(t) * k + lane];
      if (prob != nullptr) my_p = prob[static_cast<long long>(t) * k + lane];
      if (my_row < -1 || my_row >= R_cap) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
        my_row = -1;
      }
    }
    float dotp[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) dotp[j] = 0.0f;
    const uint4* xs = dot_src + static_cast<long long>(t) * vec_per_row;
    for (int c0 = 0; c0 < vec_per_row; c0 += 64) {
      const int ca = c0 + lane, cb = c0 + 32 + lane;
      const bool oka = ca < vec_per_row, okb = cb < vec_per_row;
      const uint4 xa = oka ? __ldg(xs + ca) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 xb = okb ? __ldg(xs + cb) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
      float acc[2][8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[0][i] = acc[1][i] = 0.0f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j >= k) break;
        const int row = __shfl_sync(0xFFFFFFFFu, my_row, j);
        const float pj = __shfl_sync(0xFFFFFFFFu, my_p, j);
        if (row < 0) continue;  // warp-uniform
        const uint4* rp = Yp + static_cast<long long>(row) * vec_per_row;
        const uint4 va = oka ? __ldcs(rp + ca) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 vb = okb ? __ldcs(rp + cb) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t yw[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float ylo = bf16_lo(yw[q]), yhi = bf16_hi(yw[q]);
          acc[q >> 2][2 * (q & 3)] = __fmaf_rn(pj, ylo, acc[q >> 2][2 * (q & 3)]);
          acc[q >> 2][2 * (q & 3) + 1] = __fmaf_rn(pj, yhi, acc[q >> 2][2 * (q & 3) + 1]);
          dotp[j] = __fmaf_rn(bf16_lo(xw[q]), ylo, dotp[j]);
          dotp[j] = __fmaf_rn(bf16_hi(xw[q]), yhi, dotp[j]);
        }
      }
      uint4* op = out + static_cast<long long>(t) * vec_per_row;
      if (oka)
        __stcs(op + ca, make_uint4(pack_bf16x2(acc[0][0], acc[0][1]), pack_bf16x2(acc[0][2], acc[0][3]),
                                   pack_bf16x2(acc[0][4], acc[0][5]), pack_bf16x2(acc[0][6], acc[0][7])));
      if (okb)
        __stcs(op + cb, make_uint4(pack_bf16x2(acc[1][0], acc[1][1]), pack_bf16x2(acc[1][2], acc[1][3]),
                                   pack_bf16x2(acc[1][4], acc[1][5]), pack_bf16x2(acc[1][6], acc[1][7])));
    }
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      float v = dotp[j];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
      if (lane == j) mine = v;
    }
    if (lane < k) dprob[static_cast<long long>(t) * k + lane] = my_row >= 0 ? mine : 0.0f;
  }
}

// out[t] = bf16(sum_j [prob] * Sp[row(t, j)]) (fp32 in slot order, one
// rounding: bitwise the plain combine) together with dprob[t*k+j] =
// <dot_src[t], D[row(t, j)]>. One warp per token; per pass each lane takes
// one 16-byte column group of the token's rows and issues the loads of up to
// eight slots' Sp and D rows before any arithmetic, so every warp keeps 16
// row loads in flight (the rows are gathered, one DRAM round trip each).
// Slots beyond eight are taken in further groups of eight; kMaxK (8 or 32)
// bounds k and the dot partials held in registers.
template <int kMaxK>
__global__ void __launch_bounds__(256)
combine_dot_rows_kernel(const uint4* __restrict__ Sp, const int32_t* __restrict__ row_of_slot,
                        const float* __restrict__ prob, int T, int k, int vec_per_row,
                        int R_cap, uint4* __restrict__ out, const uint4* __restrict__ dot_src,
                        const uint4* __restrict__ D, float* __restrict__ dprob,
                        int32_t* status) {
  constexpr int kGroup = 8;
  const int lane = threadIdx.x & 31;
  const int warp0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  for (int t = warp0; t < T; t += nwarps) {
    int my_row = -1;
    float my_p = 1.0f;
    if (lane < k) {
      my_row = row_of_slot[static_cast<long long>(t) * k + lane];
      if (prob != nullptr) my_p = prob[static_cast<long long>(t) * k + lane];
      if (my_row < -1 || my_row >= R_cap) {
        set_status(status, GG_ERR_DEVICE_BAD_ROW);
        my_row = -1;
      }
    }
    float dotp[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) dotp[j] = 0.0f;
    const uint4* xs = dot_src + static_cast<long long>(t) * vec_per_row;
    for (int c0 = 0; c0 < vec_per_row; c0 += 32) {
      const int c = c0 + lane;
      const bool ok = c < vec_per_row;
      const uint4 xv = ok ? __ldg(xs + c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int g0 = 0; g0 < kMaxK; g0 += kGroup) {
        if (g0 >= k) break;
        uint4 sv[kGroup], dv[kGroup];
        float pj[kGroup];
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
          const int j = g0 + i;
          const int row = __shfl_sync(0xFFFFFFFFu, my_row, j & 31);
          pj[i] = __shfl_sync(0xFFFFFFFFu, my_p, j & 31);
          const bool live = ok && j < k && row >= 0;
          const long long off = static_cast<long long>(live ? row : 0) * vec_per_row + c;
          sv[i] = live ? __ldcs(Sp + off) : make_uint4(0u, 0u, 0u, 0u);
          dv[i] = live ? __ldcs(D + off) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
          const int j = g0 + i;
          const int row = __shfl_sync(0xFFFFFFFFu, my_row, j & 31);
          if (j >= k || row < 0) continue;  // warp-uniform
          const uint32_t sw[4] = {sv[i].x, sv[i].y, sv[i].z, sv[i].w};
          const uint32_t dw[4] = {dv[i].x, dv[i].y, dv[i].z, dv[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            acc[2 * q] = __fmaf_rn(pj[i], bf16_lo(sw[q]), acc[2 * q]);
            acc[2 * q + 1] = __fmaf_rn(pj[i], bf16_hi(sw[q]), acc[2 * q + 1]);
            dotp[j] = __fmaf_rn(bf16_lo(xw[q]), bf16_lo(dw[q]), dotp[j]);
            dotp[j] = __fmaf_rn(bf16_hi(xw[q]), bf16_hi(dw[q]), dotp[j]);
          }
        }
      }
      if (ok)
        __stcs(out + static_cast<long long>(t) * vec_per_row + c,
               make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                          pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
    }
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      if (j >= k) break;
      float v = dotp[j];
#pragma unroll
      for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, m);
      if (lane == j) mine = v;
    }
    if (lane < k) dprob[static_cast<long long>(t) * k + lane] = my_row >= 0 ? mine : 0.0f;
  }
}

// Expert parallelism: owning rank and local expert of every pair.
__global__ void __launch_bounds__(256)
ep_split_ids_kernel(const int32_t* __restrict__ idx, long long n, int El, int n_ranks,
                    int32_t* __restrict__ dest, int32_t* __restrict__ local_eid,
                    int32_t* status) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int e = idx[i];
    if (e >= 0 && e < El * n_ranks) {
      const int d = e / El;
      dest[i] = d;
      local_eid[i] = e - d * El;
    } else {
      dest[i] = -1;
      local_eid[i] = -1;
      set_status(status, GG_ERR_DEVICE_BAD_EXPERT_ID);
    }
  }
}

// out[i][c] = src[index[i]][c], one thread per 32-bit element.
__global__ void __launch_bounds__(256)
gather_rows32_kernel(const uint32_t* __restrict__ src, int src_rows, int width,
                     const int32_t* __restrict__ index, long long n, uint32_t* __restrict__ out,
                     int32_t* status) {
  const long long total = n * width;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long i = t / width;
    const int c = static_cast<int>(t - i * width);
    const int r = index[i];
    uint32_t v = 0u;
    if (r >= 0 && r < src_rows)
      v = src[static_cast<long long>(r) * width + c];
    else if (r != -1)
      set_status(status, GG_ERR_DEVICE_BAD_ROW);
    out[t] = v;
  }
}

__global__ void bounded_wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the wait must give up on its own.
    (void)mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
  }
  __syncthreads();
}


}  // namespace

cudaError_t launch_permute(const gg_bf16* x, const int32_t* idx, const float* prob, int T, int H,
                           int k, int E, int P, gg_bf16* Xp, int32_t* offsets,
                           int32_t* row_of_slot, int32_t* slot_of_row, float* prob_of_row,
                           int32_t* status, int32_t* block_hist, const DeviceInfo& dev,
                           cudaStream_t stream) {
  const long long R = static_cast<long long>(T) * k;
  const long long R_cap = R + static_cast<long long>(E) * (P - 1);
  const int nb = permute_blocks(R);
  const long long ppb = permute_pairs_per_block(R);
  // scatter: warp histograms, two partial-sum rows, expert bases
  const size_t scatter_smem = sizeof(int) * (static_cast<size_t>(kWarps) * E +
                                             2 * kPermuteBlockThreads + E);
  static std::atomic<bool> smem_opt_in[kMaxDevices];  // per device; concurrent writers agree
  if (dev.device < 0 || dev.device >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaError_t err;
  if (!smem_opt_in[dev.device].load(std::memory_order_relaxed)) {
    // up to 32 x 1024 warp counts (128 KB) at E = 1024
    err = cudaFuncSetAttribute(permute_scatter_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(sizeof(int) * (static_cast<size_t>(kWarps) *
                                                                   kMaxExperts +
                                                               2 * kPermuteBlockThreads +
                                                               kMaxExperts)));
    if (err != cudaSuccess) return err;
    smem_opt_in[dev.device].store(true, std::memory_order_relaxed);
  }
  if (nb > 0) {
    permute_count_kernel<<<nb, kPermuteBlockThreads, sizeof(int) * E, stream>>>(
        idx, R, E, ppb, block_hist, status, slot_of_row, prob_of_row, R_cap);
    count_launch();
  }
  // with no routed pairs one block writes the offsets (all zero); started
  // early behind the count kernel, it waits for the histogram rows
  err = launch_early(permute_scatter_kernel, dim3(nb > 0 ? nb : 1), dim3(kPermuteBlockThreads),
                     scatter_smem, stream, idx, prob, R, E, P, ppb, nb, block_hist, offsets,
                     row_of_slot, slot_of_row, prob_of_row);
  if (err != cudaSuccess) return err;
  count_launch();
  if (R == 0) return cudaGetLastError();
  if (Xp != nullptr) {
    err = launch_gather_rows(x, row_of_slot, slot_of_row, offsets, H, k, E,
                             static_cast<int>(R_cap), T, P > 1, nullptr, Xp, status,
                             dev.sm_count, stream, /*after_maps=*/true);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const gg_bf16* src, const int32_t* row_of_slot,
                               const int32_t* slot_of_row, const int32_t* offsets, int H, int k,
                               int E, int R_cap, int T, bool has_padding, const float* prob,
                               gg_bf16* dst, int32_t* status, int sm_count,
                               cudaStream_t stream, bool after_maps) {
  if (R_cap <= 0 || T <= 0) return cudaSuccess;
  const int vec = H / 8;
  // one token per warp: the blocks, far more than fit at once, start as
  // earlier ones finish, which balances tokens whose rows load slowly
  // (measured faster than one resident wave and than two)
  long long blocks = (static_cast<long long>(T) + 7) / 8;
  const long long cap = static_cast<long long>(sm_count) * 1024;
  if (blocks > cap) blocks = cap;
  // with padding, the same launch zeroes the padding rows: warps for the
  // tokens plus one warp per 32-row group of the rows (up to the cap)
  if (has_padding) {
    const long long pad_blocks = (static_cast<long long>(R_cap) + 255) / 256;
    blocks = blocks + pad_blocks < cap ? blocks + pad_blocks : cap;
  }
  const int32_t* pad_sor = has_padding ? slot_of_row : nullptr;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  const dim3 grid(static_cast<unsigned>(blocks)), block(256);
  cudaError_t err;
  if (after_maps) {
    err = prob != nullptr
              ? launch_early(scatter_rows_scaled_kernel, grid, block, 0, stream, s4, row_of_slot,
                             prob, T, k, vec, R_cap, d4, status, pad_sor, offsets, E)
              : launch_early(scatter_rows_kernel, grid, block, 0, stream, s4, row_of_slot, T, k,
                             vec, R_cap, d4, status, pad_sor, offsets, E);
  } else {
    if (prob != nullptr)
      scatter_rows_scaled_kernel<<<grid, block, 0, stream>>>(s4, row_of_slot, prob, T, k, vec,
                                                             R_cap, d4, status, pad_sor,
                                                             offsets, E);
    else
      scatter_rows_kernel<<<grid, block, 0, stream>>>(s4, row_of_slot, T, k, vec, R_cap, d4,
                                                      status, pad_sor, offsets, E);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaSuccess;
}

cudaError_t launch_ep_split_ids(const int32_t* idx, long long n, int El, int n_ranks,
                                int32_t* dest, int32_t* local_eid, int32_t* status,
                                cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  ep_split_ids_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(idx, n, El, n_ranks, dest,
                                                                     local_eid, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_rows32(const uint32_t* src, int src_rows, int width,
                                 const int32_t* index, long long n, uint32_t* out,
                                 int32_t* status, int sm_count, cudaStream_t stream) {
  if (n <= 0 || width <= 0) return cudaSuccess;
  long long blocks = (n * width + 255) / 256;
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  gather_rows32_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(src, src_rows, width, index,
                                                                      n, out, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_zero_pad_rows(const int32_t* slot_of_row, const int32_t* offsets, int E,
                                 int R_cap, int vec_per_row, void* dst, int sm_count,
                                 cudaStream_t stream) {
  if (R_cap <= 0) return cudaSuccess;
  long long pb = (static_cast<long long>(R_cap) + 255) / 256;
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (pb > cap) pb = cap;
  zero_pad_rows_kernel<<<static_cast<int>(pb), 256, 0, stream>>>(slot_of_row, offsets, E, R_cap,
                                                                  vec_per_row,
                                                                  static_cast<uint4*>(dst));
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_combine(const gg_bf16* Yp, const int32_t* row_of_slot, const float* prob,
                           int T, int k, int H, int R_cap, gg_bf16* out, const float* rowdot,
                           int n_rowdot, const gg_bf16* dot_src, const gg_bf16* dot_rows,
                           float* dprob, int32_t* status, int sm_count, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  const int vec = H / 8;
  long long blocks = (static_cast<long long>(T) + 7) / 8;
  // 8 blocks per SM, more than fit at once (a second, partial wave; measured
  // faster than one token per warp here, unlike the row copy)
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  const int nb = static_cast<int>(blocks);
  if (dprob != nullptr && dot_src != nullptr) {
    if (dot_rows != nullptr && k <= 8)
      combine_dot_rows_kernel<8><<<nb, 256, 0, stream>>>(
          reinterpret_cast<const uint4*>(Yp), row_of_slot, prob, T, k, vec, R_cap,
          reinterpret_cast<uint4*>(out), reinterpret_cast<const uint4*>(dot_src),
          reinterpret_cast<const uint4*>(dot_rows), dprob, status);
    else if (dot_rows != nullptr)
      combine_dot_rows_kernel<32><<<nb, 256, 0, stream>>>(
          reinterpret_cast<const uint4*>(Yp), row_of_slot, prob, T, k, vec, R_cap,
          reinterpret_cast<uint4*>(out), reinterpret_cast<const uint4*>(dot_src),
          reinterpret_cast<const uint4*>(dot_rows), dprob, status);
    else if (k <= 8)
      combine_dot_kernel<8><<<nb, 256, 0, stream>>>(
          reinterpret_cast<const uint4*>(Yp), row_of_slot, prob, T, k, vec, R_cap,
          reinterpret_cast<uint4*>(out), reinterpret_cast<const uint4*>(dot_src), dprob, status);
    else
      combine_dot_kernel<32><<<nb, 256, 0, stream>>>(
          reinterpret_cast<const uint4*>(Yp), row_of_slot, prob, T, k, vec, R_cap,
          reinterpret_cast<uint4*>(out), reinterpret_cast<const uint4*>(dot_src), dprob, status);
  } else if (dprob != nullptr)
    combine_dprob_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(Yp), row_of_slot, prob, T, k, vec, R_cap,
        reinterpret_cast<uint4*>(out), rowdot, n_rowdot, dprob, status);
  else
    combine_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(Yp), row_of_slot, prob, T, k, vec, R_cap,
        reinterpret_cast<uint4*>(out), status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_bounded_wait_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  count_launch();
  return cudaGetLastError();
}

}  // namespace gg

// ---------------------------------------------------------------------------
// Permute for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a runtime whose
// memory pool owns every byte of the GPU after start-up and forbids cudaMalloc
// on its hot path, a plugin embedded in a host framework that gives it only
// pre-sized input and output buffers, or a C caller without any device
// allocator. For them gg_permute_noalloc keeps the permute's scratch (the
// status word and the per-block expert histograms) in one fixed array in
// device memory that is part of this library's image: every GPU that loads
// the library holds these bytes until the process exits.
//
// The array's host-side name is only a stand-in for the symbol, not a device
// address, so the host fetches the real address once per device with
// cudaGetSymbolAddress (on the device that is current at the first call) and
// passes that pointer to the kernels.
#include <mutex>

namespace gg {
namespace {

// status header + 128 histogram rows of 512 experts: any batch with E <= 512,
// T*k <= 1024 * floor(65536 / E) pairs above that (65,536 at E = 1024)
constexpr size_t kStaticScratchBytes = kWsHeader + (size_t(256) << 10);

static __device__ __align__(256) uint8_t g_permute_scratch[kStaticScratchBytes];

// Device address of g_permute_scratch per device ordinal, looked up on the
// first call made with that device current. Only a successful lookup is
// kept: a failed one (for instance a sticky error left by earlier work, or a
// first call made during a stream capture) is retried by the next call.
struct StaticScratchSlot {
  std::mutex mu;
  void* ptr = nullptr;
};
StaticScratchSlot g_static_scratch[kMaxDevices];

void* static_scratch_address(int device) {
  StaticScratchSlot& slot = g_static_scratch[device];
  std::lock_guard<std::mutex> lock(slot.mu);
  if (slot.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) == cudaSuccess) slot.ptr = p;
  }
  return slot.ptr;
}

}  // namespace
}  // namespace gg

extern "C" gg_status gg_permute_noalloc(const gg_bf16* x, const int32_t* idx, const float* prob,
                                        int T, int H, int k, int E, int pad_multiple,
                                        gg_bf16* Xp, int32_t* offsets, int32_t* row_of_slot,
                                        int32_t* slot_of_row, float* prob_of_row,
                                        gg_stream_t stream) {
  using namespace gg;
  if (T < 0 || H <= 0 || k <= 0 || E <= 0 || pad_multiple <= 0) return GG_ERR_INVALID_ARG;
  if (k > 32) return GG_ERR_INVALID_ARG;
  if (E > kMaxExperts || H % 64 != 0) return GG_ERR_UNSUPPORTED_SHAPE;
  const long long R_cap = static_cast<long long>(T) * k + static_cast<long long>(E) * (pad_multiple - 1);
  if (R_cap > 0x7FFFFFFFLL) return GG_ERR_UNSUPPORTED_SHAPE;
  // the same argument rules as gg_permute: Xp NULL asks for the row maps and
  // offsets only, and x is needed only when Xp is given
  if (offsets == nullptr) return GG_ERR_INVALID_ARG;
  if (T > 0 && (idx == nullptr || prob == nullptr || row_of_slot == nullptr ||
                slot_of_row == nullptr || prob_of_row == nullptr))
    return GG_ERR_INVALID_ARG;
  if (T > 0 && Xp != nullptr && x == nullptr) return GG_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(Xp) & 15u))
    return GG_ERR_MISALIGNED;
  // The batch must fit the fixed scratch: status header + one int32 per
  // (histogram block, expert).
  const size_t need = kWsHeader + sizeof(int32_t) * static_cast<size_t>(permute_blocks(
                                                        static_cast<long long>(T) * k)) * E;
  if (need > kStaticScratchBytes) return GG_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo dev;
  gg_status s = current_device(&dev);
  if (s != GG_OK) return s;
  if (dev.device < 0 || dev.device >= kMaxDevices) return GG_ERR_UNSUPPORTED_DEVICE;
  if (dev.cc_major != 10 || dev.cc_minor != 3) return GG_ERR_UNSUPPORTED_DEVICE;
  void* scratch = static_scratch_address(dev.device);
  if (scratch == nullptr) return GG_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t* status = static_cast<int32_t*>(scratch);
  // The array keeps the previous call's bytes: the status word must start at
  // zero; the histograms are fully rewritten before they are read.
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess) return GG_ERR_CUDA;
  int32_t* block_hist = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + kWsHeader);
  return launch_permute(x, idx, prob, T, H, k, E, pad_multiple, Xp, offsets, row_of_slot,
                        slot_of_row, prob_of_row, status, block_hist, dev, st) ==
                 cudaSuccess
             ? GG_OK
             : GG_ERR_CUDA;
}
