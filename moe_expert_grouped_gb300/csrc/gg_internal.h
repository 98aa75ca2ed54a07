// gg_internal.h — declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gg.h"

namespace gg {

// Workspace layout: [0, 256) status word + reserved; then the permute's
// per-block expert histograms (int32 [n_blocks][E]).
constexpr size_t kWsHeader = 256;
constexpr int kPermuteBlockThreads = 1024;
constexpr int kPermuteMaxBlocks = 128;  // histogram rows every scatter block reads
constexpr int kMaxExperts = 1024;
// Per-device host-side caches (launch attributes, device properties, the
// no-workspace permute's scratch address) are indexed by the device ordinal;
// ordinals at or above this are refused with GG_ERR_UNSUPPORTED_DEVICE.
constexpr int kMaxDevices = 64;

// The permute splits its R pairs into at most kPermuteMaxBlocks blocks of a
// whole number of 1024-pair steps (one 32-pair step per warp).
inline long long permute_pairs_per_block(long long pairs) {
  const long long per = (pairs + kPermuteMaxBlocks - 1) / kPermuteMaxBlocks;
  const long long step = kPermuteBlockThreads;
  const long long ppb = (per + step - 1) / step * step;
  return ppb > step ? ppb : step;
}

inline int permute_blocks(long long pairs) {
  const long long ppb = permute_pairs_per_block(pairs);
  return static_cast<int>((pairs + ppb - 1) / ppb);
}

void count_launch(int n = 1);

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0;
  int cc_minor = 0;
};

// Attributes of the current device (cached per device).
gg_status current_device(DeviceInfo* out);

// ------------------------------------------------------------------ gg_permute.cu
// Xp may be null: then only the row maps and offsets are produced.
cudaError_t launch_permute(const gg_bf16* x, const int32_t* idx, const float* prob, int T, int H,
                           int k, int E, int P, gg_bf16* Xp, int32_t* offsets,
                           int32_t* row_of_slot, int32_t* slot_of_row, float* prob_of_row,
                           int32_t* status, int32_t* block_hist, const DeviceInfo& dev,
                           cudaStream_t stream);

// dst[row_of_slot[t*k+j]] = src[t] (times prob[t*k+j] when prob is not
// null); with has_padding, rows below offsets[E] whose slot_of_row is -1 are
// zeroed. after_maps: the launch directly follows the kernel that writes the
// row maps, so it may start before that kernel ends (it waits for its
// results before its first access).
cudaError_t launch_gather_rows(const gg_bf16* src, const int32_t* row_of_slot,
                               const int32_t* slot_of_row, const int32_t* offsets, int H, int k,
                               int E, int R_cap, int T, bool has_padding, const float* prob,
                               gg_bf16* dst, int32_t* status, int sm_count, cudaStream_t stream,
                               bool after_maps = false);

// dprob (nullable): dprob[t*k+j] = sum_b rowdot[row_of_slot[t*k+j]][b], rows of
// rowdot (n_rowdot + 7) / 8 * 8 floats apart.
// With dot_src (and dprob): dprob[t*k+j] = <dot_src[t], D[row_of_slot[t*k+j]]>
// with D = dot_rows, or Yp when dot_rows is null.
cudaError_t launch_combine(const gg_bf16* Yp, const int32_t* row_of_slot, const float* prob,
                           int T, int k, int H, int R_cap, gg_bf16* out, const float* rowdot,
                           int n_rowdot, const gg_bf16* dot_src, const gg_bf16* dot_rows,
                           float* dprob, int32_t* status, int sm_count, cudaStream_t stream);

// dest[i] = idx[i] / El, local_eid[i] = idx[i] % El (ids in [0, El * n_ranks);
// -1 and the bad-expert status otherwise).
cudaError_t launch_ep_split_ids(const int32_t* idx, long long n, int El, int n_ranks,
                                int32_t* dest, int32_t* local_eid, int32_t* status,
                                cudaStream_t stream);

// out[i][c] = src[index[i]][c] on 32-bit elements (zero for index -1; zero and
// the bad-row status for an index outside [-1, src_rows)).
cudaError_t launch_gather_rows32(const uint32_t* src, int src_rows, int width,
                                 const int32_t* index, long long n, uint32_t* out,
                                 int32_t* status, int sm_count, cudaStream_t stream);

// Zeroes row r (vec_per_row 16-byte vectors of dst) for every r < offsets[E]
// whose slot_of_row is -1 (the padding rows).
cudaError_t launch_zero_pad_rows(const int32_t* slot_of_row, const int32_t* offsets, int E,
                                 int R_cap, int vec_per_row, void* dst, int sm_count,
                                 cudaStream_t stream);

cudaError_t launch_bounded_wait_selftest(int32_t* status, uint64_t limit_ns, cudaStream_t stream);

// ------------------------------------------------------------------ gg_gemm.cu
enum GemmMode : int {
  kFwdPlain = 0,
  kFwdSwiglu = 1,
  kDgradPlain = 2,
  kDgradSwigluBwd = 3,
  kFwdQgeglu = 4,       // kFwdSwiglu with the QuickGELU gate
  kDgradQgegluBwd = 5,  // kDgradSwigluBwd with the QuickGELU gate
};

struct GemmArgs {
  GemmMode mode;
  const gg_bf16* A;        // [R_cap][Kred] activations (K-major)
  const gg_bf16* B;        // [E][Nw][Kw] forward weight
  const int32_t* offsets;  // [E+1]
  int E, R_cap;
  int Kred;                // reduction length
  int Nout;                // accumulator columns that exist (fwd: N, dgrad: K of the weight)
  int Nw, Kw;              // forward weight dims
  gg_bf16* C;              // output
  gg_bf16* H1_save;        // fwd SwiGLU: [R_cap][2F] or null
  const gg_bf16* H1;       // dgrad SwiGLU backward: [R_cap][2F]
  const float* row_scale;  // dgrad: prob_of_row; fwd gated epilogue: the weighted
                           // activation's prob_of_row; or null
  float* rowdot = nullptr; // dgrad SwiGLU backward: [R_cap][stride] partials, or null
  int32_t* status;
  // Gathered A operand: row r of A is gather_src[slot_of_row[r] / gather_k]
  // (zero where the slot is -1); gather_src is token-major [gather_rows][Kred].
  const gg_bf16* gather_src = nullptr;
  const int32_t* slot_of_row = nullptr;
  int gather_k = 1;
  int gather_rows = 0;
};

cudaError_t launch_grouped_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                                gg_status* host_err);

// cuTensorMapEncodeTiled, fetched once through the runtime's driver entry point.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

cudaError_t launch_swiglu(const gg_bf16* H1, const int32_t* offsets, int E, int R_cap, int F,
                          float alpha, const float* row_scale, gg_bf16* A, int sm_count,
                          cudaStream_t stream);

// ------------------------------------------------------------------ gg_gemm_mx.cu
// MXFP8 grouped GEMM (layouts in gg_mx.cuh). C[r][n] = sum_k A[r][k] B[e][n][k]
// with both operands E4M3 + E8M0 scales; modes as GemmMode, the dgrad modes
// reading pre-transposed weights (B is always [E][Nw][K], K-major).
struct MxGemmArgs {
  GemmMode mode;
  const uint8_t* A;        // [R_cap][K] E4M3
  const uint8_t* As;       // A scale tiles: sf_tiles x (K/128) x 512 B
  int sf_tiles;            // scale tiles the A-scale buffer holds
  const uint8_t* B;        // [E][Nw][K] E4M3
  const uint8_t* Bs;       // weight scale tiles [E][NT][K/128][1024 B]
  const int32_t* offsets;  // [E+1]
  int E, R_cap, K, Nout, Nw;
  gg_bf16* C;              // plain modes: BF16 [R_cap][Nout]
  uint8_t* Cq;             // gated modes: E4M3 [R_cap][Kq] (fwd: A, Kq = F; bwd: dH1, Kq = 2F)
  uint8_t* Cs;             // and its scale tiles
  int Kq;
  gg_bf16* H1_save;        // gated fwd: [R_cap][2F] or null
  const gg_bf16* H1;       // gated bwd: [R_cap][2F]
  const float* row_scale;  // as GemmArgs
  float* rowdot;           // gated bwd: [R_cap][roundup8(2 NT)] partials, or null
  int32_t* status;
};

// Column tiles per row-tile pair of a mode (gated fwd: 96 gate + 96 up
// columns; otherwise 192 columns).
int mx_column_tiles(GemmMode mode, int Nout);

cudaError_t launch_grouped_gemm_mx(const MxGemmArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                                   gg_status* host_err);

// ------------------------------------------------------------------ gg_mx_quant.cu
// tiles_before[e] = sum over e' < e of ceil(rows of e' / 128), e in [0, E].
cudaError_t launch_mx_tile_prefix(const int32_t* offsets, int E, int32_t* tiles_before,
                                  cudaStream_t stream);

// Permuted MXFP8 A operand, token-ordered: every pair (t, j) with a row
// gets Q[row_of_slot[t*k+j]] = the E4M3 codes of src[t] (times prob[t*k+j],
// rounded to BF16, when prob is not null) and its scales in the 128-row tile
// of the expert e whose rows contain it (tile tiles_before[e] + local row /
// 128). Every other cell of S (sf_tiles_cap tiles of K/128 x 512 bytes) gets
// code 0: rows no pair reaches, padding rows, tiles past the last expert's.
// With has_padding the padding rows of Q are zeroed. Launched behind the
// kernel that writes tiles_before (it starts early and waits for it).
cudaError_t launch_mx_quantize_rows(const gg_bf16* src, int T, int K, int k,
                                    const int32_t* row_of_slot, const int32_t* slot_of_row,
                                    const int32_t* offsets, const int32_t* tiles_before, int E,
                                    int R_cap, bool has_padding, int sf_tiles_cap,
                                    const float* prob, uint8_t* Q, uint8_t* S, int32_t* status,
                                    int sm_count, cudaStream_t stream);

// One weight operand: Wq[e][n][k] = E4M3 of W[e][n][k] (transpose = false,
// W [E][N][K]) or of W[e][k][n] (transpose = true, W [E][K][N]), quantised
// along k; scales into the weight scale tiles of the GEMM that reads it
// (gated_F > 0: FC1's gate/up column tiles).
cudaError_t launch_mx_prepare_weight(const gg_bf16* W, int E, int N, int K, bool transpose,
                                     int gated_F, int NT, uint8_t* Wq, uint8_t* S,
                                     cudaStream_t stream);

// alpha of the gated activation of a gg_epilogue (1 for SwiGLU, 1.702 for
// QuickGeGLU), 0 for epilogues without one.
inline float glu_alpha(gg_epilogue epi) {
  switch (epi) {
    case GG_EPI_SWIGLU:
    case GG_EPI_SWIGLU_BWD:
      return 1.0f;
    case GG_EPI_QGEGLU:
    case GG_EPI_QGEGLU_BWD:
      return 1.702f;
    default:
      return 0.0f;
  }
}

}  // namespace gg
