// gg_gemm_mx.cu — the persistent grouped GEMM of the expert layer with MXFP8
// operands on the block-scaled tensor cores of sm_103a.
//
// The pages run the routed expert projections in MXFP8 (NVIDIA/Megatron-LM PR
// #7333, "Validation"; "[Main] Support paged stash with device-initiated
// GroupedLinear", NVIDIA/Megatron-LM PR #6828, "End-to-end GB300
// validation"). Both operands are E4M3 with one E8M0 scale per 32 elements
// along K (format and scale layouts: gg_mx.cuh); the product accumulates in
// FP32 in TMEM.
//
// Structure as in the BF16 grouped GEMM (gg_gemm.cu): clusters of two CTAs
// form one tcgen05 MMA pair (cta_group::2, M = 256), warp 0 is the TMA
// producer, one thread of the even CTA issues the MMAs, 8 epilogue warps per
// CTA drain TMEM. Differences:
//   * a k-step is 128 E4M3 elements (one 128-byte swizzle row): the pair's
//     A tile (2 x 128 x 128 B) and B tile (2 x 128 x 128 B) plus their scale
//     tiles (512 B of A scales per CTA, 1 KB of B scales) land on one
//     barrier; 6 stages;
//   * the scale tiles go from shared memory to TMEM with tcgen05.cp (ordered
//     before the MMAs of the same thread), then four MMAs of K = 32 each
//     pick their 32-element block with the instruction's scale ids;
//   * the MMA is 256 x 256 x 32 (a 192-column MMA costs 137 clocks against
//     128 for 256 columns, measured): one 256-column accumulator at TMEM
//     columns 0-255, the scale cells of the stages at 256 + 16 s. With a
//     single accumulator the epilogue first moves its share of it into
//     registers as BF16 (every GEMM result of the layer is BF16), releases it
//     to the MMA issuer, and only then does the activation, quantisation and
//     stores while the next tile's MMAs run. The SwiGLU backward, whose
//     epilogue bounds its kernel, instead runs 256 x 128 x 32 MMAs into two
//     128-column accumulators (columns 0-127 and 128-255), so its epilogue
//     drains half as much per tile while the MMAs fill the other one;
//   * the B operand is always K-major: the input-gradient GEMMs read weights
//     that were transposed and quantised along their output dimension once
//     (gg_mx_prepare_weights);
//   * the gated epilogues quantise what they hand to the next GEMM: FC1
//     writes H1 (BF16, for the backward) and the activation as E4M3 + scales;
//     the SwiGLU-backward epilogue writes dH1 as E4M3 + scales. A thread owns
//     one row and 32 consecutive columns per chunk, exactly one scale block,
//     so the block maximum needs no exchange between threads.
// Every wait is bounded like the BF16 kernel's.

#include <cuda_runtime.h>

#include <atomic>

#include "gg_epilogue.cuh"
#include "gg_internal.h"
#include "gg_mx.cuh"
#include "gg_ptx.cuh"

namespace gg {
namespace {

using mx::kKStep;
using mx::kTileN;
using mx::kTileNHalf;

constexpr int BM = 128;
constexpr int STAGES = 6;
constexpr int kCluster = 2;
constexpr uint16_t kClusterMask = 0x3;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 128 + 32 * kEpiWarps;  // producer, MMA, two idle, epilogue
constexpr uint32_t A_BYTES = BM * kKStep;               // 16 KB
constexpr uint32_t B_BYTES = kTileNHalf * kKStep;       // 16 KB
constexpr uint32_t AB_STAGE = A_BYTES + B_BYTES;        // 32 KB, 1024-aligned
constexpr uint32_t SF_STAGE = mx::kSfaBytes + mx::kSfbBytes;
constexpr uint32_t TX_BYTES = AB_STAGE + SF_STAGE;      // per CTA and stage (256 columns)
constexpr uint32_t TMEM_COLS = 512;

__host__ __device__ constexpr bool two_acc_mode(int mode) {
  return mode == kDgradSwigluBwd || mode == kDgradQgegluBwd;
}
__host__ __device__ constexpr int tile_cols(int mode) { return two_acc_mode(mode) ? 128 : 256; }

// TMEM columns of stage s's scale cells: A scales in 4, B scales in 8
__device__ __forceinline__ uint32_t sf_col(int stage) { return 256u + 16u * stage; }

// The expert row starts are read from the offsets in global memory (two
// cached loads per tile), which leaves room for a sixth stage.
struct SmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];   // accumulator a holds a finished tile (a = 1: two-accumulator mode)
  uint64_t tempty[2];  // the epilogue has read accumulator a
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int pad_;
  int tiles_before[kMaxExperts + 1];
  int sf_before[kMaxExperts + 1];  // first 128-row scale tile of each expert
};

constexpr uint32_t kWarpStagingBytes = 32 * 64;
constexpr uint32_t kStagingBytes = kEpiWarps * kWarpStagingBytes;
constexpr size_t kSmemBytes =
    1024 + STAGES * (AB_STAGE + SF_STAGE) + kStagingBytes + sizeof(SmemTail);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(256 + 16 * STAGES <= TMEM_COLS, "scale cells next to the accumulator");

struct MxParams {
  const int32_t* offsets;
  int E;
  int R_cap;
  int K;       // reduction length (multiple of 128)
  int Nout;    // accumulator columns that exist
  int F;       // gated modes
  int NT;      // column tiles per row-tile pair
  int NTw;     // 256-column tiles of the weight scale layout
  gg_bf16* C;  // plain modes: BF16 [R_cap][ldc]
  long long ldc;
  uint8_t* Cq;     // gated modes: E4M3 output [R_cap][Kq]
  uint8_t* Cs;     // and its 128-row scale tiles
  int Kq;
  gg_bf16* H1_save;
  const gg_bf16* H1;
  const float* row_scale;
  float* rowdot;
  int rowdot_stride;
  int32_t* status;
};

// 16-byte slot of half c (0..1) of row r (0..31) in a warp's staging buffer.
__device__ __forceinline__ int stage_slot8(int r, int c) { return r * 2 + (c ^ ((r >> 2) & 1)); }

// Warp-collective store of a 32-row x 32-byte E4M3 chunk: lane i holds row i
// in q[8]; row r goes to row0 + r * ld, rows r >= nvalid are skipped.
__device__ __forceinline__ void store_chunk8(uint4* stg, const uint32_t (&q)[8], uint8_t* row0,
                                             long long ld, int nvalid) {
  const int lane = threadIdx.x & 31;
  stg[stage_slot8(lane, 0)] = make_uint4(q[0], q[1], q[2], q[3]);
  stg[stage_slot8(lane, 1)] = make_uint4(q[4], q[5], q[6], q[7]);
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int r = 16 * j + (lane >> 1);
    const int c = lane & 1;
    const uint4 v = stg[stage_slot8(r, c)];
    if (r < nvalid) reinterpret_cast<uint4*>(row0 + r * ld)[c] = v;
  }
  __syncwarp();
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapSA,
                       const __grid_constant__ CUtensorMap mapSB, const MxParams p) {
  constexpr bool kGatedFwd = MODE == kFwdSwiglu || MODE == kFwdQgeglu;
  constexpr bool kGatedBwd = MODE == kDgradSwigluBwd || MODE == kDgradQgegluBwd;
  constexpr float kAlpha = (MODE == kFwdQgeglu || MODE == kDgradQgegluBwd) ? 1.702f : 1.0f;
  // The SwiGLU backward, whose epilogue is the slowest stage, uses 128-column
  // tiles in two accumulators (TMEM columns 0-127 and 128-255): the MMAs of
  // one tile run while the epilogue works on the other. The other modes use
  // one 256-column accumulator that the epilogue drains to registers.
  constexpr bool kTwoAcc = two_acc_mode(MODE);
  constexpr int kTN = tile_cols(MODE);        // accumulator columns per tile
  constexpr uint32_t kBRows = kTN / 2;        // weight rows per CTA
  constexpr uint32_t kTx = A_BYTES + kBRows * kKStep + mx::kSfaBytes + kTN * 4;
  static_assert(kTwoAcc || kTx == TX_BYTES, "a 256-column stage fills the whole slot");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  const uint32_t sf_base = sbase + STAGES * AB_STAGE;
  uint8_t* staging = smem + STAGES * (AB_STAGE + SF_STAGE);
  SmemTail& st = *reinterpret_cast<SmemTail*>(staging + kStagingBytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  const int NT = p.NT;
  const int KB = p.K / kKStep;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;

  if (warp == 0) {
    bool bad = false;
    int carry = 0, carry_sf = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int tiles = 0, sft = 0;
      if (e < E) {
        const int o0 = p.offsets[e];
        const int o1 = p.offsets[e + 1];
        if (o1 < o0) bad = true;
        const int mtiles = o1 > o0 ? (o1 - o0 + BM - 1) / BM : 0;
        tiles = ((mtiles + kCluster - 1) / kCluster) * NT;
        sft = mtiles;
      }
      int incl = tiles, incl_sf = sft;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        const int m = __shfl_up_sync(0xFFFFFFFFu, incl_sf, d);
        if (lane >= d) {
          incl += n;
          incl_sf += m;
        }
      }
      if (e < E) {
        st.tiles_before[e] = carry + incl - tiles;
        st.sf_before[e] = carry_sf + incl_sf - sft;
      }
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
      carry_sf += __shfl_sync(0xFFFFFFFFu, incl_sf, 31);
    }
    if (lane == 0) {
      const int o_first = p.offsets[0];
      const int o_last = p.offsets[E];
      if (o_first != 0 || o_last > p.R_cap || o_last < 0) bad = true;
      st.tiles_before[E] = carry;
      st.sf_before[E] = carry_sf;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      st.total_tiles = bad ? 0 : carry;
      st.abort_flag = 0;
      if (bad && blockIdx.x == 0) set_status(p.status, GG_ERR_DEVICE_BAD_OFFSETS);
#pragma unroll
      for (int s = 0; s < STAGES; ++s) {
        mbar_init(smem_u32(&st.full[s]), 1);
        mbar_init(smem_u32(&st.empty[s]), 1);
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(smem_u32(&st.tfull[a]), 1);
        mbar_init(smem_u32(&st.tempty[a]), kCluster * kEpiWarps);
      }
      mbar_init(smem_u32(&st.mma_done), 1);
      mbar_fence_init();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
  } else if (warp == 1) {
    tmem_alloc_pair(smem_u32(&st.tmem_base), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();

  const int cluster_id = static_cast<int>(blockIdx.x) / kCluster;
  const int n_clusters = static_cast<int>(gridDim.x) / kCluster;
  const uint32_t tmem_base = st.tmem_base;
  const int total = st.total_tiles;
  volatile int* abort_flag = &st.abort_flag;

  // Warpgroup 0 holds the producer and MMA warps (warps 2 and 3 idle),
  // warpgroups 1 and 2 the epilogue warps. In the SwiGLU-backward modes the
  // first gives registers to the other two (128 x 88 + 256 x 192 <= 384 x 168,
  // the registers of the launch), so that epilogue runs without spills.
  constexpr bool kSplitRegs = MODE == kDgradSwigluBwd || MODE == kDgradQgegluBwd;
  if (warp < 4) {
    if constexpr (kSplitRegs) asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      if (lane == 0) {
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
        tma_prefetch_desc(&mapSA);
        tma_prefetch_desc(&mapSB);
        const int h = static_cast<int>(crank);
        int stage = 0;
        uint32_t phase = 0;
        uint32_t used = 0, last_phase = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += n_clusters) {
          int e, mp, nt;
          decode_tile(tile, st.tiles_before, E, NT, e, mp, nt);
          const int mt = mp * kCluster + h;
          const int row0 = __ldg(p.offsets + e) + mt * BM;
          const int sf_row = (st.sf_before[e] + mt) * KB;
          const int b_row = kGatedFwd ? h * p.F + nt * kTileNHalf : nt * kTN + h * kBRows;
          // weight scales: the 256-column tile holding this tile's columns, and
          // for a 128-column tile the half (128 words) that covers it
          const int sfb_row = (e * p.NTw + (kTwoAcc ? nt >> 1 : nt)) * KB;
          const int sfb_x = kTwoAcc ? (nt & 1) * 128 : 0;
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait_bounded(smem_u32(&st.empty[stage]), phase ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = mapa_shared(smem_u32(&st.full[stage]), 0);
            const uint32_t sa = sbase + stage * AB_STAGE;
            const uint32_t sb = sa + A_BYTES;
            const uint32_t ssa = sf_base + stage * SF_STAGE;
            const uint32_t ssb = ssa + mx::kSfaBytes;
            if (leader) mbar_arrive_expect_tx(smem_u32(&st.full[stage]), kCluster * kTx);
            tma_load_2d_pair(sa, &mapA, fb, kb * kKStep, row0);
            tma_load_3d_pair(sb, &mapB, fb, kb * kKStep, b_row, e);
            tma_load_2d_pair(ssa, &mapSA, fb, 0, sf_row + kb);
            tma_load_2d_pair(ssb, &mapSB, fb, sfb_x, sfb_row + kb);
            used |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        for (int s = 0; s < STAGES; ++s)
          if (used & (1u << s)) {
            if (leader)
              (void)mbar_wait_bounded(smem_u32(&st.full[s]), (last_phase >> s) & 1u, nullptr,
                                      p.status);
            (void)mbar_wait_bounded(smem_u32(&st.empty[s]), (last_phase >> s) & 1u, nullptr,
                                    p.status);
          }
      }
    } else if (warp == 1) {
      if (lane == 0 && leader) {
        // ------------------------------------------------ MMA issuer (even CTA)
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = cluster_id; tile < total && ok; tile += n_clusters) {
          // the epilogue has read this accumulator's previous tile out of TMEM
          if (!mbar_wait_bounded(smem_u32(&st.tempty[acc]), acc_phase ^ 1u, abort_flag, p.status))
            break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kTN);
          for (int kb = 0; kb < KB; ++kb) {
            if (!mbar_wait_bounded(smem_u32(&st.full[stage]), phase, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + stage * AB_STAGE;
            const uint32_t sb = sa + A_BYTES;
            const uint32_t ssa = sf_base + stage * SF_STAGE;
            const uint32_t ssb = ssa + mx::kSfaBytes;
            const uint32_t tsa = tmem_base + sf_col(stage);
            const uint32_t tsb = tsa + 4;
            mx::cp_scales_pair(tsa, ssa);
            mx::cp_scales_pair(tsb, ssb);  // columns 0-127
            if (!kTwoAcc) mx::cp_scales_pair(tsb + 4, ssb + 512);  // columns 128-255
#pragma unroll
            for (int kk = 0; kk < kKStep / 32; ++kk) {
              const uint64_t adesc = make_sdesc(sa + kk * 32, 16, 1024);
              const uint64_t bdesc = make_sdesc(sb + kk * 32, 16, 1024);
              mx::mma_mx_pair(d_tmem, adesc, bdesc,
                              mx::make_idesc_mx(kCluster * BM, kTN, kk, kk), tsa, tsb,
                              (kb | kk) != 0 ? 1u : 0u);
            }
            tc_commit_pair_mc(smem_u32(&st.empty[stage]), kClusterMask);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair_mc(smem_u32(&st.tfull[acc]), kClusterMask);
          if (kTwoAcc) acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
        tc_commit_pair(smem_u32(&st.mma_done));
        (void)mbar_wait_bounded(smem_u32(&st.mma_done), 0, nullptr, p.status);
      }
    }
  } else {
    if constexpr (kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // -------------------------------------------------- epilogue (kEpiWarps warps)
    // Warp w reads TMEM lanes 32*(w%4) .. +31 (its rows); the two warps of a
    // lane quadrant take half of the 256 columns each. The warp's share goes
    // to registers as BF16 (acc[16] = 4 chunks of 32 columns), the warp
    // reports the accumulator free, then works from registers.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    const int r = q * 32 + lane;
    constexpr int kChunks = kTN / 64;  // 32-column chunks of this warp per tile
    int eacc = 0;                      // accumulator of the current tile
    uint32_t acc_phase = 0;
    uint4* stg = reinterpret_cast<uint4*>(staging + (warp - 4) * kWarpStagingBytes);
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    for (int tile = cluster_id; tile < total; tile += n_clusters) {
      int e, mp, nt;
      decode_tile(tile, st.tiles_before, E, NT, e, mp, nt);
      const int mt = mp * kCluster + static_cast<int>(crank);
      const long long tile_row0 = static_cast<long long>(__ldg(p.offsets + e)) + mt * BM;
      const long long grow = tile_row0 + r;
      const long long row_end = __ldg(p.offsets + e + 1);
      const bool valid = grow < row_end;
      const long long grow0 = grow - lane;
      const int nvalid = static_cast<int>(max(0LL, min(32LL, row_end - grow0)));
      // the 128-row scale tile (e, mt) is written by the tile that owns it:
      // every row of it, code 0 for the rows past the expert's end
      const bool owns_sf = tile_row0 < row_end;
      const long long sf_tile = st.sf_before[e] + mt;
      // the four 32-column chunks of this warp: plain and backward modes take
      // columns [128 half, +128); FC1 takes gate [64 half, +64) and the
      // matching up columns [128 + 64 half, +64)
      float scale = 1.0f;
      if (MODE == kDgradPlain && p.row_scale != nullptr && valid) scale = p.row_scale[grow];
      // the saved H1 does not depend on the accumulator: fetch the first
      // chunk of the backward before waiting for the MMAs
      const int Fb = p.Nout;
      const int n0 = nt * kTN;
      const int cb0 = half * (kTN / 2);
      const gg_bf16* hrow0 = kGatedBwd ? p.H1 + grow0 * (2LL * Fb) + n0 : nullptr;
      uint4 graw[4], uraw[4];
      if (kGatedBwd && n0 + cb0 < Fb) {
        load_chunk_raw(graw, hrow0 + cb0, 2LL * Fb, nvalid);
        load_chunk_raw(uraw, hrow0 + Fb + cb0, 2LL * Fb, nvalid);
      }
      if (!mbar_wait_bounded(smem_u32(&st.tfull[eacc]), acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      uint4 acc[kChunks][4];
#pragma unroll
      for (int j = 0; j < kChunks; ++j) {
        const int col = kGatedFwd ? (j < 2 ? 64 * half + 32 * j : 128 + 64 * half + 32 * (j - 2))
                                  : cb0 + 32 * j;
        float v[32];
        tmem_ld32(tq + static_cast<uint32_t>(eacc * kTN + col), v);
        pack_bf16x32(v, scale, acc[j]);
      }
      tc_fence_before();
      __syncwarp();
      // this warp's share of the accumulator is in registers: the MMAs of a
      // later tile may overwrite it (relaxed arrive: only the completed TMEM
      // reads need ordering)
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&st.tempty[eacc]), 0));
      if (kTwoAcc) eacc ^= 1;
      if (eacc == 0) acc_phase ^= 1u;

      if constexpr (MODE == kFwdPlain || MODE == kDgradPlain) {
        gg_bf16* crow0 = p.C + grow0 * p.ldc + n0;
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int c = cb0 + 32 * j;
          if (n0 + c < p.Nout) store_chunk(stg, acc[j], crow0 + c, p.ldc, nvalid);
        }
      } else if constexpr (kGatedFwd) {
        const int F = p.F;
        const bool scaled = p.row_scale != nullptr;
        const float prow = scaled && valid ? p.row_scale[grow] : 1.0f;
        const int j0 = nt * kTileNHalf;
        const int KGq = p.Kq / kKStep;
        gg_bf16* hrow = p.H1_save + grow0 * (2LL * F) + j0;
        uint8_t* arow0 = p.Cq + grow0 * p.Kq + j0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = 64 * half + 32 * j;  // gate column in the tile's 128
          if (j0 + c >= F) break;
          if (p.H1_save != nullptr) {
            store_chunk(stg, acc[j], hrow + c, 2LL * F, nvalid);
            store_chunk(stg, acc[j + 2], hrow + F + c, 2LL * F, nvalid);
          }
          uint32_t pa[16];  // the activation as BF16 pairs
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t gw[4] = {acc[j][i].x, acc[j][i].y, acc[j][i].z, acc[j][i].w};
            const uint32_t uw[4] = {acc[j + 2][i].x, acc[j + 2][i].y, acc[j + 2][i].z,
                                    acc[j + 2][i].w};
#pragma unroll
            for (int w = 0; w < 4; ++w)
              pa[4 * i + w] =
                  pack_bf16x2(glu_mul(bf16_lo(gw[w]), bf16_lo(uw[w]), kAlpha, scaled, prow),
                              glu_mul(bf16_hi(gw[w]), bf16_hi(uw[w]), kAlpha, scaled, prow));
          }
          uint32_t qv[8];
          const uint32_t code = mx::quantize32_bf16(pa, qv);
          store_chunk8(stg, qv, arow0 + c, p.Kq, nvalid);
          if (owns_sf) {
            const int col = j0 + c;
            p.Cs[(sf_tile * KGq + col / kKStep) * mx::kSfaBytes + mx::sf_byte(r, (col >> 5) & 3)] =
                static_cast<uint8_t>(valid ? code : 0u);
          }
        }
      } else {  // gated backward: dA columns n0 + cb0.., output [dg | du] quantised, K = 2F
        const int F = Fb;
        float prs = 1.0f;
        if (p.row_scale != nullptr && valid) prs = p.row_scale[grow];
        const int c_end = min(cb0 + kTN / 2, F - n0);  // multiple of 32
        const int KGq = p.Kq / kKStep;
        uint8_t* drow0 = p.Cq + grow0 * p.Kq + n0;
        // four independent partial sums: rd[c & 1] takes column pair c, .x its
        // low and .y its high column
        float2 rd[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        constexpr bool kAlphaOne = kAlpha == 1.0f;
        const bool want_dot = p.rowdot != nullptr;
#pragma unroll
        for (int j = 0; j < kChunks; ++j) {
          const int c = cb0 + 32 * j;
          if (c >= c_end) break;
          uint4 gw[4], uw[4];
          transpose_chunk(stg, graw, gw);
          transpose_chunk(stg, uraw, uw);
          if (c + 32 < c_end) {
            load_chunk_raw(graw, hrow0 + c + 32, 2LL * F, nvalid);
            load_chunk_raw(uraw, hrow0 + F + c + 32, 2LL * F, nvalid);
          }
          uint32_t as[16], gs[16], us[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            as[4 * i + 0] = acc[j][i].x; as[4 * i + 1] = acc[j][i].y;
            as[4 * i + 2] = acc[j][i].z; as[4 * i + 3] = acc[j][i].w;
            gs[4 * i + 0] = gw[i].x; gs[4 * i + 1] = gw[i].y;
            gs[4 * i + 2] = gw[i].z; gs[4 * i + 3] = gw[i].w;
            us[4 * i + 0] = uw[i].x; us[4 * i + 1] = uw[i].y;
            us[4 * i + 2] = uw[i].z; us[4 * i + 3] = uw[i].w;
          }
          // column pairs as packed fp32 pairs (the same rounding per column as
          // the scalar form); dg and du leave as the BF16 pairs the block
          // quantiser takes
          uint32_t pg[16], pu[16];
          if (want_dot) {
#pragma unroll
            for (int hh = 0; hh < 16; ++hh)
              glu_mul_bwd2<true, kAlphaOne>(make_float2(bf16_lo(as[hh]), bf16_hi(as[hh])), prs,
                                            gs[hh], us[hh], kAlpha, pg[hh], pu[hh], rd[hh & 1]);
          } else {
#pragma unroll
            for (int hh = 0; hh < 16; ++hh)
              glu_mul_bwd2<false, kAlphaOne>(make_float2(bf16_lo(as[hh]), bf16_hi(as[hh])), prs,
                                             gs[hh], us[hh], kAlpha, pg[hh], pu[hh], rd[hh & 1]);
          }
          uint32_t qv[8];
          const uint32_t code_g = mx::quantize32_bf16(pg, qv);
          store_chunk8(stg, qv, drow0 + c, p.Kq, nvalid);
          const uint32_t code_u = mx::quantize32_bf16(pu, qv);
          store_chunk8(stg, qv, drow0 + F + c, p.Kq, nvalid);
          if (owns_sf) {
            const int cg = n0 + c, cu = F + n0 + c;
            p.Cs[(sf_tile * KGq + cg / kKStep) * mx::kSfaBytes + mx::sf_byte(r, (cg >> 5) & 3)] =
                static_cast<uint8_t>(valid ? code_g : 0u);
            p.Cs[(sf_tile * KGq + cu / kKStep) * mx::kSfaBytes + mx::sf_byte(r, (cu >> 5) & 3)] =
                static_cast<uint8_t>(valid ? code_u : 0u);
          }
        }
        if (p.rowdot != nullptr && valid)
          p.rowdot[grow * p.rowdot_stride + nt * 2 + half] =
              (rd[0].x + rd[1].x) + (rd[0].y + rd[1].y);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  cluster_sync();
}

// ------------------------------------------------------------------ host side

bool encode_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int rank,
                const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box,
                CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = fn(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims,
                        strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch_mx_mode(const CUtensorMap (&maps)[4], const MxParams& kp,
                           const DeviceInfo& dev, cudaStream_t stream) {
  // (atomic: host threads may launch concurrently; every writer stores the same value)
  static std::atomic<int> clusters_for[kMaxDevices];
  if (dev.device < 0 || dev.device >= kMaxDevices) return cudaErrorInvalidDevice;
  const int d = dev.device;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (clusters_for[d].load(std::memory_order_relaxed) == 0) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_mx_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(static_cast<unsigned>((dev.sm_count / kCluster) * kCluster), 1, 1);
    e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_mx_kernel<MODE>, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    clusters_for[d].store(n < dev.sm_count / kCluster ? n : dev.sm_count / kCluster,
                          std::memory_order_relaxed);
  }
  cfg.gridDim = dim3(
      static_cast<unsigned>(clusters_for[d].load(std::memory_order_relaxed) * kCluster), 1, 1);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_mx_kernel<MODE>, maps[0], maps[1],
                                           maps[2], maps[3], kp);
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int mx_column_tiles(GemmMode mode, int Nout) {
  const bool gated = mode == kFwdSwiglu || mode == kFwdQgeglu;
  const int tn = tile_cols(mode);
  return gated ? (Nout / 2 + kTileNHalf - 1) / kTileNHalf : (Nout + tn - 1) / tn;
}

cudaError_t launch_grouped_gemm_mx(const MxGemmArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                                   gg_status* host_err) {
  *host_err = GG_OK;
  CUtensorMap maps[4];
  const int KB = a.K / kKStep;
  const int NT = mx_column_tiles(a.mode, a.Nout);
  // the weight scale tiles are laid out per 256 columns in every mode
  const bool gated_fwd = a.mode == kFwdSwiglu || a.mode == kFwdQgeglu;
  const int NTw = gated_fwd ? NT : (a.Nout + kTileN - 1) / kTileN;
  const bool two_acc = two_acc_mode(a.mode);
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.R_cap)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.K)};
    const cuuint32_t box[2] = {kKStep, BM};
    if (!encode_map(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.A, 2, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B)) {
      *host_err = GG_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.K), static_cast<cuuint64_t>(a.Nw),
                                static_cast<cuuint64_t>(a.E)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.K),
                                   static_cast<cuuint64_t>(a.K) * a.Nw};
    const cuuint32_t box[3] = {kKStep, two_acc ? kTileNHalf / 2u : kTileNHalf, 1};
    if (!encode_map(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.B, 3, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_128B)) {
      *host_err = GG_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  {
    // A scales: [sf_tiles * KB] rows of 128 words (512 B)
    const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(a.sf_tiles) * KB};
    const cuuint64_t strides[1] = {mx::kSfaBytes};
    const cuuint32_t box[2] = {128, 1};
    if (!encode_map(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, a.As, 2, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_NONE)) {
      *host_err = GG_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  {
    // B scales: [E * NTw * KB] rows of 256 words (1 KB); a 128-column tile
    // loads the half that covers it
    const cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(a.E) * NTw * KB};
    const cuuint64_t strides[1] = {mx::kSfbBytes};
    const cuuint32_t box[2] = {two_acc ? 128u : 256u, 1};
    if (!encode_map(&maps[3], CU_TENSOR_MAP_DATA_TYPE_UINT32, a.Bs, 2, dims, strides, box,
                    CU_TENSOR_MAP_SWIZZLE_NONE)) {
      *host_err = GG_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  MxParams kp{};
  kp.offsets = a.offsets;
  kp.E = a.E;
  kp.R_cap = a.R_cap;
  kp.K = a.K;
  kp.Nout = a.Nout;
  kp.NT = NT;
  kp.NTw = NTw;
  kp.C = a.C;
  kp.Cq = a.Cq;
  kp.Cs = a.Cs;
  kp.Kq = a.Kq;
  kp.H1_save = a.H1_save;
  kp.H1 = a.H1;
  kp.row_scale = a.row_scale;
  kp.rowdot = a.rowdot;
  kp.rowdot_stride = (2 * NT + 7) / 8 * 8;
  kp.status = a.status;
  switch (a.mode) {
    case kFwdPlain:
      kp.ldc = a.Nout;
      return launch_mx_mode<kFwdPlain>(maps, kp, dev, stream);
    case kDgradPlain:
      kp.ldc = a.Nout;
      return launch_mx_mode<kDgradPlain>(maps, kp, dev, stream);
    case kFwdSwiglu:
      kp.F = a.Nout / 2;
      return launch_mx_mode<kFwdSwiglu>(maps, kp, dev, stream);
    case kFwdQgeglu:
      kp.F = a.Nout / 2;
      return launch_mx_mode<kFwdQgeglu>(maps, kp, dev, stream);
    case kDgradSwigluBwd:
      kp.F = a.Nout;
      return launch_mx_mode<kDgradSwigluBwd>(maps, kp, dev, stream);
    case kDgradQgegluBwd:
      kp.F = a.Nout;
      return launch_mx_mode<kDgradQgegluBwd>(maps, kp, dev, stream);
  }
  *host_err = GG_ERR_INVALID_ARG;
  return cudaErrorInvalidValue;
}

}  // namespace gg
