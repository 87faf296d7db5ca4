// Device helpers of the bit-plane scans (plane words -> token prefixes -> floats,
// and the cp.async staging ring), shared by scan.cu and scan_heads.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace fathom {
namespace bitplane {

template <int SH>
__device__ __forceinline__ uint32_t shift_signed(uint32_t x) {
  // SH > 0: right shift, SH < 0: left shift (compile-time)
  if constexpr (SH > 0) return x >> SH;
  else if constexpr (SH < 0) return x << (-SH);
  else return x;
}

// bit select: bits of a where mask is set, of b elsewhere
__device__ __forceinline__ uint32_t bitsel(uint32_t mask, uint32_t a, uint32_t b) { return (a & mask) | (b & ~mask); }

// o_k for depth DEP: nibble m holds the prefix of token 4m+k in its top DEP bits
// (plane 0 in bit 3); bits below the prefix are left unspecified (masked later).
template <int DEP, int K>
__device__ __forceinline__ uint32_t nibble_word(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
  const uint32_t s0 = shift_signed<K - 3>(w0);
  if constexpr (DEP == 1) return s0;
  const uint32_t s1 = shift_signed<K - 2>(w1);
  if constexpr (DEP == 2) return bitsel(0x88888888u, s0, s1);
  const uint32_t s2 = shift_signed<K - 1>(w2);
  if constexpr (DEP == 3) return bitsel(0x88888888u, s0, bitsel(0x44444444u, s1, s2));
  const uint32_t s3 = shift_signed<K>(w3);
  return bitsel(0x88888888u, s0, bitsel(0x44444444u, s1, bitsel(0x22222222u, s2, s3)));
}

// One token's prefix as the float 1 + u/16: the byte 0x80 | u<<3 (u = the
// token's 4-bit nibble, low bits below the prefix cleared) placed under the
// exponent byte 0x3F gives 0x3F800000 | u<<19 (exact).  `bytes` holds four
// such bytes, the selector picks byte J.
template <int J>
__device__ __forceinline__ float prefix_float(uint32_t bytes) {
  return __uint_as_float(__byte_perm(bytes, 0x3F000000u, 0x7044u | (J << 8)));
}

template <int BYTES>
__device__ __forceinline__ void cp_async(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(s), "l"(gmem), "n"(BYTES) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace bitplane
}  // namespace fathom
