// gg_gemm.cu — the persistent grouped GEMM of the expert layer on sm_103a.
//
// One launch covers every expert ("perf(moe): add frozen grouped GEMM for
// adapter training", AlignmentResearch/Megatron-LM PR #3, "Why this change":
// one grouped kernel instead of one small GEMM per expert). Per-expert row
// counts are read from the device-resident offsets array (NVIDIA/Megatron-LM
// PR #7333, "Summary": device metadata, no host synchronisation).
//
// Design (one CTA per SM, clusters of two CTAs = one tcgen05 MMA pair,
// 320 threads per CTA, warp-specialised):
//   warp 0     TMA producer in each CTA: its own 128 rows of A (128 x 64) and
//              its half of the B tile (128 x 64 of 256 x 64), BF16 with
//              128-byte swizzle, into a 6-stage ring (32 KB per stage); the
//              loads of both CTAs complete on the even CTA's barrier;
//   warp 1     allocates 512 TMEM columns in both CTAs (two 128 x 256 fp32
//              accumulators each); in the even CTA one lane issues
//              tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) over the
//              pair's shared memory and multicasts its commits to both CTAs;
//   warps 2-9  epilogue in each CTA: tcgen05.ld of its 128 accumulator rows
//              (one TMEM lane = one output row per thread, two warps per lane
//              quadrant splitting the columns), fused SwiGLU / SwiGLU-backward
//              / probability scale, BF16 stores masked to the expert's rows;
//              then each warp reports the accumulator free to the even CTA.
// Per SM and 64-deep K step the pair moves 32 KB into shared memory for a
// 128 x 256 x 64 product (a single-CTA 128 x 256 tile needs 48 KB), which
// halves the per-SM weight traffic and leaves room for a deeper ring.
// The two accumulators let the epilogue of tile i overlap the MMAs of tile
// i+1. Work items are (expert, 256-row pair of row blocks, 256-column block),
// enumerated expert-major with the column block fastest and dealt
// round-robin to clusters; CTA rank r takes row block 2*pair+r. A row block
// that runs past its expert's last row reads the next expert's rows (or TMA
// zero fill past R_cap) and those rows are simply not stored: every output
// row depends only on its own input row and its expert's weight (bitwise
// batch invariance).
//
// The dgrad variants read the forward weight [E][N][K] as an N-contiguous
// ("MN-major") B operand straight from its forward layout, so no transposed
// copy of the frozen weights exists.
//
// Every wait is bounded (gg_ptx.cuh); a wait that runs out records
// GG_ERR_DEVICE_TIMEOUT, raises a CTA-wide abort flag, and the CTA drains its
// in-flight TMA loads and MMAs, frees TMEM and exits after a final cluster
// barrier (so no CTA leaves while its peer may still write into it).

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "gg_epilogue.cuh"
#include "gg_internal.h"
#include "gg_ptx.cuh"

namespace gg {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int kCluster = 2;  // the two CTAs of one MMA pair
constexpr uint16_t kClusterMask = 0x3;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue
constexpr uint32_t A_BYTES = BM * BK * 2;               // 16 KB: this CTA's A rows
constexpr uint32_t B_HALF_BYTES = (BN / 2) * BK * 2;     // 16 KB: this CTA's half of B
constexpr uint32_t STAGE_BYTES = A_BYTES + B_HALF_BYTES;  // per CTA and stage
constexpr uint32_t TMEM_COLS = 512;

struct SmemTail {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int pad_;
  int tiles_before[kMaxExperts + 1];
  int row_start[kMaxExperts + 1];
};

// Each epilogue warp owns a 2 KB staging buffer (32 rows x 32 BF16) used to
// turn row-per-lane results into row-contiguous global stores and loads.
constexpr uint32_t kWarpStagingBytes = 32 * 64;
constexpr uint32_t kStagingBytes = kEpiWarps * kWarpStagingBytes;
constexpr size_t kSmemBytes = 1024 + STAGES * STAGE_BYTES + kStagingBytes + sizeof(SmemTail);
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct KParams {
  const int32_t* offsets;
  int E;
  int R_cap;
  int Kred;
  int Nout;
  int F;
  int NT;
  gg_bf16* C;
  long long ldc;
  gg_bf16* H1_save;
  const gg_bf16* H1;
  const float* row_scale;
  float* rowdot;               // dgrad SwiGLU backward: [R_cap][rowdot_stride] partial <acc, a>
  int rowdot_stride;
  int32_t* status;
  const int32_t* slot_of_row;  // gathered A: source row of every permuted row
  int gather_k;
  int gather_rows;             // rows of the gather source; this index reads zeros
};

template <int MODE, bool GATHER>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                    const __grid_constant__ CUtensorMap mapB, const KParams p) {
  // gated epilogues: act(g) * u with act(g) = g * sigmoid(kAlpha * g)
  constexpr bool kGatedFwd = MODE == kFwdSwiglu || MODE == kFwdQgeglu;
  constexpr bool kGatedBwd = MODE == kDgradSwigluBwd || MODE == kDgradQgegluBwd;
  constexpr bool kDgrad = MODE == kDgradPlain || kGatedBwd;
  constexpr float kAlpha = (MODE == kFwdQgeglu || MODE == kDgradQgegluBwd) ? 1.702f : 1.0f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;  // 1024-aligned: required by the 128B swizzle
  SmemTail& st = *reinterpret_cast<SmemTail*>(smem + STAGES * STAGE_BYTES + kStagingBytes);
  // The SwiGLU-backward GEMM keeps one stage fewer in flight: its epilogue's
  // saved-H1 loads then compete with fewer operand loads (measured 1.4-2.3 %
  // faster with 5 stages, 3.7 % slower with 4; the other modes lose 2-4 %
  // with 5).
  constexpr int kStagesUsed =
      (MODE == kDgradSwigluBwd || MODE == kDgradQgegluBwd) ? STAGES - 1 : STAGES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int E = p.E;
  const int NT = p.NT;
  const int KB = p.Kred / BK;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;

  // ---- tile table from the device offsets (warp 0), TMEM (warp 1)
  if (warp == 0) {
    bool bad = false;
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int tiles = 0;
      if (e < E) {
        const int o0 = p.offsets[e];
        const int o1 = p.offsets[e + 1];
        if (o1 < o0) bad = true;
        const int mtiles = (o1 - o0 + BM - 1) / BM;
        tiles = o1 > o0 ? ((mtiles + kCluster - 1) / kCluster) * NT : 0;
        st.row_start[e] = o0;
      }
      int incl = tiles;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += n;
      }
      if (e < E) st.tiles_before[e] = carry + incl - tiles;
      carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (lane == 0) {
      const int o_first = p.offsets[0];
      const int o_last = p.offsets[E];
      if (o_first != 0 || o_last > p.R_cap || o_last < 0) bad = true;
      st.row_start[E] = o_last;
      st.tiles_before[E] = carry;
    }
    bad = __any_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
      st.total_tiles = bad ? 0 : carry;
      st.abort_flag = 0;
      if (bad && blockIdx.x == 0) set_status(p.status, GG_ERR_DEVICE_BAD_OFFSETS);
#pragma unroll
      for (int s = 0; s < kStagesUsed; ++s) {
        mbar_init(smem_u32(&st.full[s]), 1);   // even CTA: its producer's expect_tx
        mbar_init(smem_u32(&st.empty[s]), 1);  // the pair's MMA commit
      }
      for (int a = 0; a < 2; ++a) {
        mbar_init(smem_u32(&st.tfull[a]), 1);
        mbar_init(smem_u32(&st.tempty[a]), kCluster * kEpiWarps);  // every epilogue warp
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
  // Both CTAs' barriers must be initialised before any load, commit or
  // arrive of the pair can target them.
  cluster_sync();

  const int cluster_id = static_cast<int>(blockIdx.x) / kCluster;
  const int n_clusters = static_cast<int>(gridDim.x) / kCluster;
  const uint32_t tmem_base = st.tmem_base;
  const int total = st.total_tiles;
  volatile int* abort_flag = &st.abort_flag;

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    // Lane 0 waits for free stages, arms the barrier and loads B; A is loaded
    // by lane 0 as one box, or, when gathered, by all 32 lanes as four-row
    // gathers of the token rows each permuted row stands for.
    if (lane == 0) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB);
    }
    const int h = static_cast<int>(crank);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t used = 0, last_phase = 0;
    bool ok = true;
    for (int tile = cluster_id; tile < total && ok; tile += n_clusters) {
      int e, mp, nt;
      decode_tile(tile, st.tiles_before, E, NT, e, mp, nt);
      const int row0 = st.row_start[e] + (mp * kCluster + h) * BM;
      int src[4] = {0, 0, 0, 0};
      if (GATHER) {
        const int row_end = st.row_start[e + 1];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = row0 + 4 * lane + i;
          const int slot = r < row_end ? p.slot_of_row[r] : -1;
          src[i] = slot >= 0 ? slot / p.gather_k : p.gather_rows;  // past the end: zero fill
        }
      }
      if (!GATHER && lane != 0) continue;
      for (int kb = 0; kb < KB; ++kb) {
        int free_ok = 1;
        if (lane == 0)
          free_ok = mbar_wait_bounded(smem_u32(&st.empty[stage]), phase ^ 1u, abort_flag, p.status)
                        ? 1
                        : 0;
        if (GATHER) free_ok = __shfl_sync(0xFFFFFFFFu, free_ok, 0);
        if (!free_ok) {
          ok = false;
          break;
        }
        const uint32_t fb = mapa_shared(smem_u32(&st.full[stage]), 0);
        const uint32_t sa = sbase + stage * STAGE_BYTES;
        const uint32_t sb = sa + A_BYTES;
        if (lane == 0) {
          // the even CTA's barrier counts the bytes of both CTAs' loads
          if (leader) mbar_arrive_expect_tx(smem_u32(&st.full[stage]), kCluster * STAGE_BYTES);
          if (!GATHER) tma_load_2d_pair(sa, &mapA, fb, kb * BK, row0);
          if (MODE == kFwdPlain) {
            tma_load_3d_pair(sb, &mapB, fb, kb * BK, nt * BN + h * (BN / 2), e);
          } else if (kGatedFwd) {
            // half 0: gate rows j0.., half 1: up rows F + j0..
            tma_load_3d_pair(sb, &mapB, fb, kb * BK, h * p.F + nt * (BN / 2), e);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_3d_pair(sb + j * (B_HALF_BYTES / 2), &mapB, fb,
                               nt * BN + h * (BN / 2) + 64 * j, kb * BK, e);
          }
        }
        if (GATHER) {
          __syncwarp();  // the barrier is armed before any lane's gather lands
          tma_gather4_pair(sa + lane * 4 * 128, &mapA, fb, kb * BK, src[0], src[1], src[2],
                           src[3]);
        }
        used |= 1u << stage;
        last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
        if (++stage == kStagesUsed) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Before the CTA may exit, the pair's MMAs must have consumed (and so
    // the loads must have landed in) every stage this producer filled.
    if (lane == 0)
      for (int s = 0; s < kStagesUsed; ++s)
        if (used & (1u << s)) {
          if (leader)
            (void)mbar_wait_bounded(smem_u32(&st.full[s]), (last_phase >> s) & 1u, nullptr,
                                    p.status);
          (void)mbar_wait_bounded(smem_u32(&st.empty[s]), (last_phase >> s) & 1u, nullptr,
                                  p.status);
        }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (even CTA)
      constexpr bool kMN = kDgrad;
      constexpr uint32_t idesc = make_idesc_bf16(kCluster * BM, BN, kMN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = cluster_id; tile < total && ok; tile += n_clusters) {
        if (!mbar_wait_bounded(smem_u32(&st.tempty[acc]), acc_phase ^ 1u, abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded(smem_u32(&st.full[stage]), phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t adesc = make_sdesc(sa + kk * 32, 16, 1024);
            const uint64_t bdesc = kMN ? make_sdesc(sb + kk * 2048, B_HALF_BYTES / 2, 1024)
                                       : make_sdesc(sb + kk * 32, 16, 1024);
            tc_mma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          // the stage is free in both CTAs once these MMAs have read it
          tc_commit_pair_mc(smem_u32(&st.empty[stage]), kClusterMask);
          if (++stage == kStagesUsed) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(smem_u32(&st.tfull[acc]), kClusterMask);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs of the pair must retire before TMEM is freed.
      tc_commit_pair(smem_u32(&st.mma_done));
      (void)mbar_wait_bounded(smem_u32(&st.mma_done), 0, nullptr, p.status);
    }
  } else {
    // -------------------------------------------------- epilogue (kEpiWarps warps)
    // Warp w may only read TMEM lanes 32*(w%4) .. +31: two warps share each
    // lane quadrant and split the tile's columns in halves.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = cluster_id; tile < total; tile += n_clusters) {
      int e, mp, nt;
      decode_tile(tile, st.tiles_before, E, NT, e, mp, nt);
      const int mt = mp * kCluster + static_cast<int>(crank);
      const long long grow = static_cast<long long>(st.row_start[e]) + mt * BM + r;
      const bool valid = grow < st.row_start[e + 1];
      // the warp's 32 rows are consecutive: row 0 is grow0, rows < nvalid exist
      const long long grow0 = grow - lane;
      const int nvalid = static_cast<int>(
          max(0LL, min(32LL, static_cast<long long>(st.row_start[e + 1]) - grow0)));
      uint4* stg = reinterpret_cast<uint4*>(smem + STAGES * STAGE_BYTES +
                                            (warp - 2) * kWarpStagingBytes);
      if (MODE == kFwdPlain || MODE == kDgradPlain) {
        float scale = 1.0f;
        if (MODE == kDgradPlain && p.row_scale != nullptr && valid) scale = p.row_scale[grow];
        const int n0 = nt * BN;
        const int c0 = half * (BN / 2);
        gg_bf16* crow0 = p.C + grow0 * p.ldc + n0;
        if (!mbar_wait_bounded(smem_u32(&st.tfull[acc]), acc_phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
#pragma unroll 1
        for (int c = c0; c < c0 + BN / 2; c += 32) {
          if (n0 + c >= p.Nout) break;
          float v[32];
          tmem_ld32(tbase + c, v);
          uint4 w[4];
          pack_bf16x32(v, scale, w);
          store_chunk(stg, w, crow0 + c, p.ldc, nvalid);
        }
      } else if (kGatedFwd) {
        const int F = p.F;
        constexpr float alpha = kAlpha;
        const bool scaled = p.row_scale != nullptr;  // weighted activation
        const float prow = scaled && valid ? p.row_scale[grow] : 1.0f;
        const int j0 = nt * (BN / 2);
        const int c0 = half * (BN / 4);
        gg_bf16* arow0 = p.C + grow0 * F + j0;
        gg_bf16* hrow0 = p.H1_save + grow0 * (2LL * F) + j0;
        if (!mbar_wait_bounded(smem_u32(&st.tfull[acc]), acc_phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
#pragma unroll 1
        for (int c = c0; c < c0 + BN / 4; c += 32) {
          if (j0 + c >= F) break;
          float g[32], u[32];
          tmem_ld32(tbase + c, g);
          tmem_ld32(tbase + BN / 2 + c, u);
          uint4 w[4];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            g[i] = round_bf16(g[i]);
            u[i] = round_bf16(u[i]);
          }
          if (p.H1_save != nullptr) {
            pack_bf16x32(g, 1.0f, w);
            store_chunk(stg, w, hrow0 + c, 2LL * F, nvalid);
            pack_bf16x32(u, 1.0f, w);
            store_chunk(stg, w, hrow0 + F + c, 2LL * F, nvalid);
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) g[i] = glu_mul(g[i], u[i], alpha, scaled, prow);
          pack_bf16x32(g, 1.0f, w);
          store_chunk(stg, w, arow0 + c, F, nvalid);
        }
      } else {  // gated backward: F = Nout, output row [dg | du] of width 2F
        const int F = p.Nout;
        float scale = 1.0f;
        if (p.row_scale != nullptr && valid) scale = p.row_scale[grow];
        const int n0 = nt * BN;
        const int c0 = half * (BN / 2);
        const int c_end = min(c0 + BN / 2, F - n0);  // multiple of 32 (F % 64 == 0)
        const gg_bf16* hrow0 = p.H1 + grow0 * (2LL * F) + n0;
        gg_bf16* drow0 = p.C + grow0 * (2LL * F) + n0;
        // The saved H1 does not depend on the accumulator: fetch the first
        // chunk before waiting for the MMAs, then always one chunk ahead.
        uint4 graw[4], uraw[4];
        if (c0 < c_end) {
          load_chunk_raw(graw, hrow0 + c0, 2LL * F, nvalid);
          load_chunk_raw(uraw, hrow0 + F + c0, 2LL * F, nvalid);
        }
        if (!mbar_wait_bounded(smem_u32(&st.tfull[acc]), acc_phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
        // this row's <acc, a> over this warp's columns, in four independent
        // partial sums (a single 32-long chain per chunk would serialise):
        // rd[c & 1] takes column pair c, .x its low and .y its high column
        float2 rd[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
        const bool want_dot = p.rowdot != nullptr;
        constexpr float alpha = kAlpha;
        constexpr bool kAlphaOne = kAlpha == 1.0f;
#pragma unroll 1
        for (int c = c0; c < c_end; c += 32) {
          float v[32];
          tmem_ld32(tbase + c, v);
          uint4 gw[4], uw[4];
          transpose_chunk(stg, graw, gw);
          transpose_chunk(stg, uraw, uw);
          if (c + 32 < c_end) {
            load_chunk_raw(graw, hrow0 + c + 32, 2LL * F, nvalid);
            load_chunk_raw(uraw, hrow0 + F + c + 32, 2LL * F, nvalid);
          }
          uint32_t gs[16], us[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            gs[4 * i + 0] = gw[i].x; gs[4 * i + 1] = gw[i].y;
            gs[4 * i + 2] = gw[i].z; gs[4 * i + 3] = gw[i].w;
            us[4 * i + 0] = uw[i].x; us[4 * i + 1] = uw[i].y;
            us[4 * i + 2] = uw[i].z; us[4 * i + 3] = uw[i].w;
          }
          // column pairs as packed fp32 pairs: half the multiply-add
          // instructions of the scalar form, the same rounding per column
          uint32_t dgw[16], duw[16];
          if (want_dot) {
#pragma unroll
            for (int h = 0; h < 16; ++h)
              glu_mul_bwd2<true, kAlphaOne>(make_float2(v[2 * h], v[2 * h + 1]), scale, gs[h],
                                            us[h], alpha, dgw[h], duw[h], rd[h & 1]);
          } else {
#pragma unroll
            for (int h = 0; h < 16; ++h)
              glu_mul_bwd2<false, kAlphaOne>(make_float2(v[2 * h], v[2 * h + 1]), scale, gs[h],
                                             us[h], alpha, dgw[h], duw[h], rd[h & 1]);
          }
          uint4 w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w[i] = make_uint4(dgw[4 * i], dgw[4 * i + 1], dgw[4 * i + 2], dgw[4 * i + 3]);
          store_chunk(stg, w, drow0 + c, 2LL * F, nvalid);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w[i] = make_uint4(duw[4 * i], duw[4 * i + 1], duw[4 * i + 2], duw[4 * i + 3]);
          store_chunk(stg, w, drow0 + F + c, 2LL * F, nvalid);
        }
        if (p.rowdot != nullptr && valid)
          p.rowdot[grow * p.rowdot_stride + nt * 2 + half] =
              (rd[0].x + rd[1].x) + (rd[0].y + rd[1].y);
      }
      tc_fence_before();
      __syncwarp();
      // this warp's share of the accumulator is free: tell the MMA issuer. The
      // arrive is relaxed: a release would first wait for this warp's
      // output stores (measured 3.5 % of FC2 and dgrad FC2), and the barrier
      // only has to order the completed TMEM reads.
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&st.tempty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
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

// Standalone gated activation over rows [0, offsets[E]) — same arithmetic as
// the fused FC1 epilogue (glu_mul on the BF16 values of g and u).
__global__ void __launch_bounds__(256)
swiglu_kernel(const uint4* __restrict__ H1, const int32_t* __restrict__ offsets, int E, int F,
              float alpha, const float* __restrict__ row_scale, uint4* __restrict__ A) {
  const bool scaled = row_scale != nullptr;
  const long long rows = offsets[E];
  const int vec = F / 8;
  const long long n = rows * vec;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / vec;
    const int c = static_cast<int>(i - r * vec);
    const uint4 gw = __ldg(H1 + r * (2LL * vec) + c);
    const uint4 uw = __ldg(H1 + r * (2LL * vec) + vec + c);
    const uint32_t gs[4] = {gw.x, gw.y, gw.z, gw.w};
    const uint32_t us[4] = {uw.x, uw.y, uw.z, uw.w};
    const float pr = scaled ? row_scale[r] : 1.0f;
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
      o[h] = pack_bf16x2(glu_mul(bf16_lo(gs[h]), bf16_lo(us[h]), alpha, scaled, pr),
                         glu_mul(bf16_hi(gs[h]), bf16_hi(us[h]), alpha, scaled, pr));
    A[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ------------------------------------------------------------------ host side

bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  EncodeTiledFn fn = encode_tiled_fn();
  if (fn == nullptr) return false;
  cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                        const_cast<void*>(base), dims, strides_bytes, box, elem_strides,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int MODE, bool GATHER>
cudaError_t launch_mode(const CUtensorMap& ma, const CUtensorMap& mb, const KParams& kp,
                        const DeviceInfo& dev, cudaStream_t stream) {
  // Per device: the shared-memory opt-in and the number of clusters that can
  // be resident at once (the grid is persistent: one cluster per SM pair).
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
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, GATHER>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(static_cast<unsigned>((dev.sm_count / kCluster) * kCluster), 1, 1);
    e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<MODE, GATHER>, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    clusters_for[d].store(n < dev.sm_count / kCluster ? n : dev.sm_count / kCluster,
                          std::memory_order_relaxed);
  }
  cfg.gridDim = dim3(
      static_cast<unsigned>(clusters_for[d].load(std::memory_order_relaxed) * kCluster), 1, 1);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE, GATHER>, ma, mb, kp);
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, const DeviceInfo& dev, cudaStream_t stream,
                                gg_status* host_err) {
  *host_err = GG_OK;
  CUtensorMap ma, mb;
  const bool gather = a.gather_src != nullptr;
  {
    // Direct: box of 128 rows over A[R_cap][Kred]. Gathered: one-row box over
    // the token-major source, loaded four rows at a time.
    const cuuint64_t rows = gather ? static_cast<cuuint64_t>(a.gather_rows) : a.R_cap;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.Kred), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.Kred) * 2};
    const cuuint32_t box[2] = {BK, gather ? 1u : static_cast<cuuint32_t>(BM)};
    if (!encode_bf16_map(&ma, gather ? a.gather_src : a.A, 2, dims, strides, box)) {
      *host_err = GG_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.Kw), static_cast<cuuint64_t>(a.Nw),
                                static_cast<cuuint64_t>(a.E)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.Kw) * 2,
                                   static_cast<cuuint64_t>(a.Kw) * a.Nw * 2};
    cuuint32_t box[3] = {BK, BN / 2, 1};  // each CTA of a pair loads half of B
    if (a.mode == kDgradPlain || a.mode == kDgradSwigluBwd || a.mode == kDgradQgegluBwd)
      box[1] = 64;
    if (!encode_bf16_map(&mb, a.B, 3, dims, strides, box)) {
      *host_err = GG_ERR_CUDA;
      return cudaErrorInvalidValue;
    }
  }
  KParams kp{};
  kp.offsets = a.offsets;
  kp.E = a.E;
  kp.R_cap = a.R_cap;
  kp.Kred = a.Kred;
  kp.Nout = a.Nout;
  kp.C = a.C;
  kp.H1_save = a.H1_save;
  kp.H1 = a.H1;
  kp.row_scale = a.row_scale;
  kp.rowdot = a.rowdot;
  kp.rowdot_stride = (2 * ((a.Nout + BN - 1) / BN) + 7) / 8 * 8;
  kp.status = a.status;
  kp.slot_of_row = a.slot_of_row;
  kp.gather_k = a.gather_k;
  kp.gather_rows = a.gather_rows;
  switch (a.mode) {
    case kFwdPlain:
      kp.F = 0;
      kp.NT = (a.Nout + BN - 1) / BN;
      kp.ldc = a.Nout;
      return gather ? launch_mode<kFwdPlain, true>(ma, mb, kp, dev, stream)
                    : launch_mode<kFwdPlain, false>(ma, mb, kp, dev, stream);
    case kFwdSwiglu:
    case kFwdQgeglu:
      kp.F = a.Nout / 2;
      kp.NT = (kp.F + BN / 2 - 1) / (BN / 2);
      kp.ldc = kp.F;
      if (a.mode == kFwdQgeglu)
        return gather ? launch_mode<kFwdQgeglu, true>(ma, mb, kp, dev, stream)
                      : launch_mode<kFwdQgeglu, false>(ma, mb, kp, dev, stream);
      return gather ? launch_mode<kFwdSwiglu, true>(ma, mb, kp, dev, stream)
                    : launch_mode<kFwdSwiglu, false>(ma, mb, kp, dev, stream);
    case kDgradPlain:
      kp.F = 0;
      kp.NT = (a.Nout + BN - 1) / BN;
      kp.ldc = a.Nout;
      return gather ? launch_mode<kDgradPlain, true>(ma, mb, kp, dev, stream)
                    : launch_mode<kDgradPlain, false>(ma, mb, kp, dev, stream);
    case kDgradSwigluBwd:
    case kDgradQgegluBwd:
      kp.F = a.Nout;
      kp.NT = (a.Nout + BN - 1) / BN;
      kp.ldc = 2LL * a.Nout;
      if (a.mode == kDgradQgegluBwd)
        return gather ? launch_mode<kDgradQgegluBwd, true>(ma, mb, kp, dev, stream)
                      : launch_mode<kDgradQgegluBwd, false>(ma, mb, kp, dev, stream);
      return gather ? launch_mode<kDgradSwigluBwd, true>(ma, mb, kp, dev, stream)
                    : launch_mode<kDgradSwigluBwd, false>(ma, mb, kp, dev, stream);
  }
  *host_err = GG_ERR_INVALID_ARG;
  return cudaErrorInvalidValue;
}

cudaError_t launch_swiglu(const gg_bf16* H1, const int32_t* offsets, int E, int R_cap, int F,
                          float alpha, const float* row_scale, gg_bf16* A, int sm_count,
                          cudaStream_t stream) {
  if (R_cap <= 0) return cudaSuccess;
  const long long n = static_cast<long long>(R_cap) * (F / 8);
  long long blocks = (n + 255) / 256;
  const long long cap = static_cast<long long>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  swiglu_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const uint4*>(H1), offsets, E, F, alpha, row_scale,
      reinterpret_cast<uint4*>(A));
  count_launch();
  return cudaGetLastError();
}

}  // namespace gg
