// gg_mx.cuh — MXFP8 building blocks shared by the quantisers and the
// block-scaled grouped GEMM (device code and layout constants).
//
// Format (NVIDIA/Megatron-LM PR #7333, "Validation": routed expert
// projections in MXFP8; the pages do not define the encoding, the OCP
// microscaling format is the reading): FP8 E4M3 elements, one E8M0 scale
// 2^e per 32 consecutive elements along a GEMM's reduction dimension. The
// scale is the smallest power of two at which the block's largest magnitude
// is at most 448 (no element saturates), e in [-127, 127]; elements are
// v * 2^-e rounded to nearest-even E4M3.
//
// Scale-factor layouts. The block-scaled tcgen05.mma (kind::mxf8f6f4,
// scale_vec::1X) reads the scale of A row m (0..127 of a CTA) from TMEM lane
// m, column base + m/32, and the scale of B column n (0..N-1 of the pair)
// from lane n%32 of the reading row's lane quadrant, column base + n/32; the
// byte inside the 32-bit cell is the instruction's scale id (the 32-element
// block of the 128-deep K step). tcgen05.cp 32x128b.warpx4 copies a 512-byte
// shared-memory tile into 32 lanes x 4 columns of every lane quadrant, so a
// 128-row (or 128-column) tile of scales is stored as
//     byte(r, b) = (r % 32) * 16 + (r / 32) * 4 + b,   b = block in the K step,
// for every 128-deep K step ("scale tile", 512 bytes). A-operand scales are
// kept per expert-local 128-row tile: tile t of expert e is scale block
// tiles_before(e) + t, and block `blk` of a K = 128*KG operand starts at
// byte (blk * KG + kg) * 512. B-operand (weight) scales are kept per GEMM
// column tile: [E][NT][KG][1024 bytes], columns 0..127 of the 256-column
// tile in the first 512 bytes and 128..255 in the second.
#pragma once

#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gg_ptx.cuh"

namespace gg {
namespace mx {

constexpr int kBlock = 32;        // elements per scale
constexpr int kRowTile = 128;     // rows per A-operand scale tile
constexpr int kKStep = 128;       // K elements (bytes) per GEMM k-step = 4 scale blocks
constexpr int kTileN = 256;       // output columns per CTA-pair tile
constexpr int kTileNHalf = 128;   // weight rows per CTA
constexpr int kSfaBytes = 512;    // one 128-row scale tile of one k-step
constexpr int kSfbBytes = 1024;   // the 256-column scale tile of one k-step

__host__ __device__ constexpr int sf_byte(int r, int b) { return (r & 31) * 16 + (r >> 5) * 4 + b; }

// Byte of column n (0..255) of a weight scale tile.
__host__ __device__ constexpr int sfb_byte(int n, int b) { return (n >> 7) * 512 + sf_byte(n & 127, b); }

// The exponent e of a block's scale from the block's largest magnitude
// (quantize32 gives the rule) and the exact factor 2^-e.
__device__ __forceinline__ int block_exponent(float amax, float& inv) {
  const uint32_t bits = __float_as_uint(amax);
  const int biased = static_cast<int>(bits >> 23);
  int e = biased == 0 ? -127 : biased - 135 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  e = e < -127 ? -127 : e;  // finite inputs give e <= 120
  inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  return e;
}

// Quantise one 32-element block. Returns the E8M0 byte (e + 127) and packs the
// E4M3 codes into q[8] (element i in byte i % 4 of word i / 4). The exponent
// comes from the bits of max|v|: with max|v| = 1.f * 2^p, the smallest e with
// max|v| / 2^e <= 448 = 1.75 * 2^8 is p - 8, plus one when 1.f > 1.75.
// A zero or subnormal maximum takes e = -127. Multiplying by 2^-e is exact;
// the conversion rounds to nearest even and saturates at 448.
__device__ __forceinline__ uint32_t quantize32(const float (&v)[32], uint32_t (&q)[8]) {
  // block maximum as a 5-level tree (a 32-long chain would serialise)
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(v[i]), fabsf(v[i + 16]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  }
  float inv;
  const int e = block_exponent(m[0], inv);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * w] * inv, v[4 * w + 1] * inv), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(v[4 * w + 2] * inv, v[4 * w + 3] * inv), __NV_SATFINITE, __NV_E4M3);
    q[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return static_cast<uint32_t>(e + 127);
}

// quantize32 of a block held as BF16 pairs (element 2i in the low half of
// p[i], 2i + 1 in the high half): the same codes and scale as quantize32 on
// the BF16 values, with half the live registers.
__device__ __forceinline__ uint32_t quantize32_bf16(const uint32_t (&p)[16], uint32_t (&q)[8]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    m[i] = fmaxf(fmaxf(fabsf(__uint_as_float(p[i] << 16)), fabsf(__uint_as_float(p[i] & 0xFFFF0000u))),
                 fmaxf(fabsf(__uint_as_float(p[i + 8] << 16)),
                       fabsf(__uint_as_float(p[i + 8] & 0xFFFF0000u))));
#pragma unroll
  for (int w = 4; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  }
  float inv;
  const int e = block_exponent(m[0], inv);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t a = p[2 * w], b = p[2 * w + 1];
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__uint_as_float(a << 16) * inv, __uint_as_float(a & 0xFFFF0000u) * inv),
        __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__uint_as_float(b << 16) * inv, __uint_as_float(b & 0xFFFF0000u) * inv),
        __NV_SATFINITE, __NV_E4M3);
    q[w] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return static_cast<uint32_t>(e + 127);
}

// quantize32 of a block spread over four neighbouring lanes (lanes 4g..4g+3
// of a warp, eight elements each as the BF16 pairs of w, each element times
// p rounded to BF16 when kScale): the four exchange their maxima, then each
// converts its own eight elements into q (element i in byte i % 4 of word
// i / 4). Returns the block's E8M0 byte. All 32 lanes must take part.
template <bool kScale>
__device__ __forceinline__ uint32_t quantize8x4(uint4 w, float p, uint2& q) {
  float v[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
  if (kScale) {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = round_bf16(v[i] * p);
  }
  float m = fmaxf(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))),
                  fmaxf(fmaxf(fabsf(v[4]), fabsf(v[5])), fmaxf(fabsf(v[6]), fabsf(v[7]))));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  float inv;
  const int e = block_exponent(m, inv);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = __nv_cvt_float2_to_fp8x2(make_float2(v[2 * i] * inv, v[2 * i + 1] * inv),
                                    __NV_SATFINITE, __NV_E4M3);
  q = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  return static_cast<uint32_t>(e + 127);
}

// Instruction descriptor, kind::mxf8f6f4 with E4M3 A and B, K-major both,
// FP32 accumulator and E8M0 scales:
//   [4,6) B scale id   [7,10) A format (0 = E4M3)   [10,13) B format
//   [17,23) N >> 3     [23] scale format (1 = E8M0)  [24,29) M >> 4
//   [29,31) A scale id
__host__ __device__ constexpr uint32_t make_idesc_mx(int M, int N, int a_sf, int b_sf) {
  return (static_cast<uint32_t>(b_sf) << 4) | ((static_cast<uint32_t>(N) >> 3) << 17) | (1u << 23) |
         ((static_cast<uint32_t>(M) >> 4) << 24) | (static_cast<uint32_t>(a_sf) << 29);
}

// D (+)= (A * 2^sfa) (B * 2^sfb)^T over one 32-deep K step, CTA pair (M = 256).
__device__ __forceinline__ void mma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 512-byte scale tile (32 rows x 16 bytes, no swizzle) from this CTA's shared
// memory into 32 lanes x 4 columns of every lane quadrant of its TMEM, for
// both CTAs of the pair (issued by the even CTA).
__device__ __forceinline__ void cp_scales_pair(uint32_t taddr, uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 16;  // 8-row core matrices 128 B apart
  d |= static_cast<uint64_t>(128u >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d)
               : "memory");
}

}  // namespace mx
}  // namespace gg
