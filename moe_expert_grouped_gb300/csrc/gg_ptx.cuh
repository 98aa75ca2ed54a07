// gg_ptx.cuh — inline-PTX wrappers for the sm_103a building blocks used by the
// grouped GEMM: mbarriers with bounded waits, TMA tensor loads, and the
// tcgen05 tensor-core path (TMEM allocation, MMA, commit, TMEM loads).
// Descriptor bit layouts follow the public PTX ISA (tcgen05 "Matrix
// Descriptors" and "Instruction descriptor" tables).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "../../include/gg.h"

namespace gg {

// Bounded waits: a wait gives up after this many nanoseconds of %globaltimer
// (or this many polls), records GG_ERR_DEVICE_TIMEOUT and lets the kernel
// wind down instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint32_t kWaitMaxPolls = 1u << 28;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialisation may start while
// the kernel ahead of it in the stream is still running. grid_dependency_wait
// returns once that kernel has completed and its writes are visible (at once
// without such a predecessor); grid_dependents_launch lets the next kernel's
// blocks be scheduled before this one ends.

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed. Returns false if
// the CTA-wide abort flag is raised or the wait ran past its limit (then the
// status word gets GG_ERR_DEVICE_TIMEOUT and the abort flag is raised).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag,
                                                  int32_t* status,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kWaitMaxPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) break;
    }
  }
  set_status(status, GG_ERR_DEVICE_TIMEOUT);
  if (abort_flag != nullptr) *abort_flag = 1;
  return false;
}

// ----------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Gather of four rows (r0..r3) of a 2-D tensor, columns [c0, c0 + box width),
// into four consecutive box rows at dst; completion is counted on an mbarrier
// of either CTA of the MMA pair. The tensor map's box is one row high.
__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int c0, int r0, int r1,
                                                 int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(cluster_bar)
      : "memory");
}

// ----------------------------------------------------------------- tcgen05

// Shared-memory matrix descriptor (64 bit):
//   [0,14)  start address >> 4      [16,30) leading-dim byte offset >> 4
//   [32,46) stride-dim byte offset >> 4   [46,48) version = 1
//   [49,52) base offset = 0          [52] LBO mode = 0
//   [61,64) layout: 2 = 128-byte swizzle
// K-major, 128B swizzle: rows of 64 BF16 (128 B), 8-row atoms 1024 B apart
// (SBO); LBO unused. MN-major, 128B swizzle: each K row holds 64 MN elements
// (128 B), 8-row groups along K are SBO apart, 64-element groups along MN are
// LBO apart.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo_bytes,
                                               uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16 with BF16 A/B and FP32 D:
//   [4,6) D format (1 = F32)  [7,10) A format (1 = BF16)  [10,13) B format
//   [15] A major (0 = K)      [16] B major (0 = K, 1 = MN)
//   [17,23) N >> 3            [24,29) M >> 4
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((static_cast<uint32_t>(N) >> 3) << 17) | ((static_cast<uint32_t>(M) >> 4) << 24);
}

// All tcgen05 instructions of the grouped GEMM use .cta_group::2: the two CTAs
// of a cluster form one MMA pair (M = 256 rows, 128 per CTA). Allocation,
// relinquish and deallocation are performed collectively by one warp of each
// CTA of the pair; MMAs and commits are issued by one thread of the even CTA.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem of both CTAs] (+)= A[256 x 16, 128 rows per CTA] * B[N x 16, N/2 rows
// per CTA]^T; the descriptors address the same shared-memory offsets in both.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at this offset in every CTA of `cta_mask` when
// all earlier tcgen05 ops of this thread finish.
__device__ __forceinline__ void tc_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

// Arrive once on this CTA's mbarrier when all earlier tcgen05 ops finish.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Address of this CTA's shared variable `local` inside CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its cluster address (possibly another CTA's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// The same arrive without release semantics: it does not wait for this
// thread's earlier global stores to become visible. For barriers that only
// order tcgen05 accesses (the TMEM reads of the epilogue, already complete
// after tcgen05.wait::ld and ordered by tcgen05.fence::before_thread_sync)
// and pass no data through memory.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// Loads into this CTA's shared memory whose completion is counted on an
// mbarrier of either CTA of the MMA pair (`cluster_bar` from mapa_shared).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(cluster_bar)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane
// (quadrant base + i), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ----------------------------------------------------------------- math

// Gated activation act(g) * u = (g * sigmoid(alpha * g)) * u in fp32, times
// the row's probability when `scaled` (the weighted activation). alpha = 1 is
// SwiGLU (alpha * g is then exactly g), 1.702 QuickGeGLU. Shared by the fused
// FC1 epilogue and the standalone kernel (same translation unit, same
// instructions), so both round alike. The sigmoid uses the fast exponential
// and divide intrinsics: their relative error (a few fp32 ulp) is far below
// the BF16 rounding applied to every result.
__device__ __forceinline__ float glu_mul(float g, float u, float alpha, bool scaled, float p) {
  const float s = __fdividef(1.0f, 1.0f + __expf(-(alpha * g)));
  const float v = (g * s) * u;
  return scaled ? v * p : v;
}

__device__ __forceinline__ float round_bf16(float x);

// Backward of act(g) * u at dA = acc * scale, act(g) = g * s with
// s = sigmoid(alpha * g): dg = dA * u * s * (1 + alpha * g * (1 - s)),
// du = dA * g * s. With kDot also dot += acc * bf16(act(g) * u): the
// unweighted activation output of the forward pass (same sigmoid and
// products as glu_mul, so the same BF16 value) against the unscaled
// accumulator, for the routing-probability gradient.
template <bool kDot>
__device__ __forceinline__ void glu_mul_bwd(float acc, float scale, float g, float u, float alpha,
                                            float& dg, float& du, float& dot) {
  const float dA = acc * scale;
  const float s = __fdividef(1.0f, 1.0f + __expf(-(alpha * g)));
  const float dact = s * (1.0f + (alpha * g) * (1.0f - s));
  const float gs = g * s;
  dg = (dA * u) * dact;
  du = dA * gs;
  if (kDot) dot = fmaf(acc, round_bf16(gs * u), dot);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi);
__device__ __forceinline__ float bf16_lo(uint32_t w);
__device__ __forceinline__ float bf16_hi(uint32_t w);

// glu_mul_bwd for two neighbouring columns at once: g and u arrive as BF16
// pairs (column 2i in the low half), dg and du leave as BF16 pairs. The
// multiplies and adds run as packed fp32 pairs (one instruction for both
// columns; each lane rounds exactly as the scalar operation would), the
// exponential and reciprocal per column with the same intrinsics as
// glu_mul, so the activation value paired with the accumulator for the
// probability gradient is bitwise the forward's. With kDot, dot.x and dot.y
// accumulate acc * bf16(act(g) * u) of the low and high column.
template <bool kDot, bool kAlphaOne>
__device__ __forceinline__ void glu_mul_bwd2(float2 acc, float scale, uint32_t gw, uint32_t uw,
                                             float alpha, uint32_t& dg, uint32_t& du,
                                             float2& dot) {
  const float2 one = make_float2(1.0f, 1.0f);
  const float2 g = make_float2(bf16_lo(gw), bf16_hi(gw));
  const float2 u = make_float2(bf16_lo(uw), bf16_hi(uw));
  const float2 dA = __fmul2_rn(acc, make_float2(scale, scale));
  const float2 ag = kAlphaOne ? g : __fmul2_rn(make_float2(alpha, alpha), g);
  const float2 y = __fadd2_rn(one, make_float2(__expf(-ag.x), __expf(-ag.y)));
  const float2 s = make_float2(__fdividef(1.0f, y.x), __fdividef(1.0f, y.y));
  const float2 om = __ffma2_rn(s, make_float2(-1.0f, -1.0f), one);  // 1 - s
  const float2 dact = __fmul2_rn(s, __ffma2_rn(ag, om, one));       // s (1 + ag (1 - s))
  const float2 gs = __fmul2_rn(g, s);
  const float2 dg2 = __fmul2_rn(__fmul2_rn(dA, u), dact);
  const float2 du2 = __fmul2_rn(dA, gs);
  dg = pack_bf16x2(dg2.x, dg2.y);
  du = pack_bf16x2(du2.x, du2.y);
  if (kDot) {
    const float2 a = __fmul2_rn(gs, u);
    const uint32_t aw = pack_bf16x2(a.x, a.y);
    dot = __ffma2_rn(acc, make_float2(bf16_lo(aw), bf16_hi(aw)), dot);
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float round_bf16(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

}  // namespace gg
