// fp32 contractions on the tcgen05 tensor cores: kind::tf32 with a two-term split.
//
// Every fp32 operand x is carried as hi = tf32(x) and lo = tf32(x - hi) (round to nearest),
// both exact tf32 values held in fp32 words. A product is taken as
//   a.b ~ a_hi.b_hi + a_hi.b_lo + a_lo.b_hi,
// three kind::tf32 MMAs into one fp32 TMEM accumulator. The dropped a_lo.b_lo term and the
// rounding of lo leave a relative error of about 2^-21 per product, against 2^-11 for a
// single tf32 pass. An operand that is exact in tf32 (bf16 input, for instance) has lo = 0
// and its two lo-terms are skipped.
//
// Operand tiles are staged by the CTA's threads with plain loads (any stride, transposed
// when the contraction index is not the contiguous one), split, and written to shared
// memory in the canonical K-major 128-byte-swizzle layout: rows of 32 fp32 of K (128 B),
// 8-row atoms of 1024 B, a tile of R rows and K elements stored as K/32 panels of R x 128 B.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "sm100.cuh"

namespace tree {
namespace tc32 {

using namespace sm100;

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// x -> (hi, lo) as fp32 bit patterns of tf32 values.
__device__ __forceinline__ void split(float x, uint32_t& hi, uint32_t& lo) {
  hi = to_tf32(x);
  lo = to_tf32(x - __uint_as_float(hi));
}

// Byte offset of element (r, k) in a K-major SW128 tile of R rows.
template <int R>
__device__ __forceinline__ uint32_t sw_off(int r, int k) {
  return static_cast<uint32_t>((k >> 5) * (R * 128) + r * 128 + ((((k & 31) >> 2) ^ (r & 7)) << 4) + ((k & 3) << 2));
}

// Splits 4 consecutive K elements of row r and writes them (hi, lo) with one 16-byte store each.
template <int R>
__device__ __forceinline__ void put4(uint8_t* hi, uint8_t* lo, int r, int k, float4 x) {
  uint4 h, l;
  split(x.x, h.x, l.x);
  split(x.y, h.y, l.y);
  split(x.z, h.z, l.z);
  split(x.w, h.w, l.w);
  const uint32_t o = sw_off<R>(r, k);
  *reinterpret_cast<uint4*>(hi + o) = h;
  *reinterpret_cast<uint4*>(lo + o) = l;
}

template <int R>
__device__ __forceinline__ void put1(uint8_t* hi, uint8_t* lo, int r, int k, float x) {
  uint32_t h, l;
  split(x, h, l);
  const uint32_t o = sw_off<R>(r, k);
  *reinterpret_cast<uint32_t*>(hi + o) = h;
  *reinterpret_cast<uint32_t*>(lo + o) = l;
}

__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// Instruction descriptor, kind::tf32 A/B (K-major), fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                                // D format fp32
         | (2u << 7)                              // A format tf32
         | (2u << 10)                             // B format tf32
         | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[M x N] (+)= A[M x K] . B[N x K]^T from split K-major SW128 tiles (A of M rows, B of N
// rows), issued by one thread. `accumulate` = 0 starts D afresh. a_lo_zero / b_lo_zero skip
// the terms of an operand whose lo part is zero.
template <int M, int N, int K>
__device__ __forceinline__ void mma3(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                     uint32_t accumulate, bool a_lo_zero = false, bool b_lo_zero = false) {
  static_assert(M == 128 && N % 16 == 0 && N >= 16 && N <= 256 && K % 32 == 0, "tile shape");
  constexpr uint32_t idesc = idesc_tf32(M, N);
#pragma unroll
  for (int s = 0; s < K / 8; ++s) {
    const uint32_t oa = (s >> 2) * (M * 128) + (s & 3) * 32, ob = (s >> 2) * (N * 128) + (s & 3) * 32;
    const uint64_t ah = desc_sw128(a_hi + oa, 16, 1024), bh = desc_sw128(b_hi + ob, 16, 1024);
    mma_tf32(d_tmem, ah, bh, idesc, (accumulate || s > 0) ? 1u : 0u);
    if (!b_lo_zero) mma_tf32(d_tmem, ah, desc_sw128(b_lo + ob, 16, 1024), idesc, 1u);
    if (!a_lo_zero) mma_tf32(d_tmem, desc_sw128(a_lo + oa, 16, 1024), bh, idesc, 1u);
  }
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

}  // namespace tc32
}  // namespace tree
