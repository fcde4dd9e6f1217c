// Device helpers of the deconstruction step shared by the split kernels and
// the fused narrow-N kernel: the row (column) exponent, and the power-of-two
// scaling with round-half-even to an integer, all as integer bit arithmetic
// on the fp64 pattern ([TME4] abstract: operands are scaled, rounded and
// reduced modulo each modulus; no fp64 arithmetic is used here).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace ozemu {

// round-half-even(x 2^s) + 2^62 for the finite double with bit pattern `bits`
// (|result - 2^62| <= 2^62 is guaranteed by the row shift).  Non-finite -> 0.
__device__ __forceinline__ uint64_t scaled_offset(uint64_t bits, int s) {
  uint32_t E = static_cast<uint32_t>(bits >> 52) & 0x7FFu;
  uint64_t mant = bits & 0xFFFFFFFFFFFFFull;
  int e0 = -1074;
  if (E != 0) {
    mant |= 1ull << 52;
    e0 = static_cast<int>(E) - 1075;
  }
  if (E == 0x7FFu) mant = 0;
  uint64_t q = 0;
  if (mant != 0) {
    int sh = e0 + s;
    if (sh >= 0) {
      q = mant << sh;
    } else {
      int d = -sh;
      d = d > 63 ? 63 : d;
      q = mant >> d;
      uint64_t rem = mant & ((1ull << d) - 1ull);
      uint64_t half = 1ull << (d - 1);
      q += static_cast<uint64_t>((rem > half) | ((rem == half) & (q & 1ull)));
    }
  }
  int64_t v = (bits >> 63) ? -static_cast<int64_t>(q) : static_cast<int64_t>(q);
  return static_cast<uint64_t>(v + (1ll << 62));
}

// frexp exponent of the double with (non-negative, nonzero) bit pattern b.
__device__ __forceinline__ int frexp_exp_bits(uint64_t b) {
  uint32_t E = static_cast<uint32_t>(b >> 52);
  if (E) return static_cast<int>(E) - 1022;
  return (64 - __clzll(static_cast<long long>(b))) - 1074;
}

template <int kThreads>
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* red) {
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  uint64_t m = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = red[w] > m ? red[w] : m;
  return m;
}

// Widest vector load a row of X allows: 2 = 32 bytes (X 32-byte aligned,
// ldx a multiple of 4), 1 = 16 bytes, 0 = single elements.
__device__ __forceinline__ int row_vector_width(const double* X, long long ldx) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(X);
  if ((a & 31u) == 0 && (ldx & 3) == 0) return 2;
  if ((a & 15u) == 0 && (ldx & 1) == 0) return 1;
  return 0;
}

// Elements k0 .. k0+7 of a row (zeros past k).  With 32-byte loads the
// warp's two load instructions each fill whole 32-byte sectors (each lane's
// eight elements are 64 bytes apart from its neighbour's).
__device__ __forceinline__ void load8_f64(const double* rowp, int k, int k0, int vec, uint64_t (&b)[8],
                                          bool last_use) {
  if (vec == 2 && k0 + 8 <= k) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      unsigned long long x0, x1, x2, x3;
      asm volatile("ld.global.nc.v4.u64 {%0, %1, %2, %3}, [%4];"
                   : "=l"(x0), "=l"(x1), "=l"(x2), "=l"(x3)
                   : "l"(rowp + k0 + 4 * q));
      b[4 * q] = x0;
      b[4 * q + 1] = x1;
      b[4 * q + 2] = x2;
      b[4 * q + 3] = x3;
    }
  } else if (vec >= 1 && k0 + 8 <= k) {
    const double2* p = reinterpret_cast<const double2*>(rowp + k0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      double2 v = last_use ? __ldcs(p + q) : __ldg(p + q);
      b[2 * q] = static_cast<uint64_t>(__double_as_longlong(v.x));
      b[2 * q + 1] = static_cast<uint64_t>(__double_as_longlong(v.y));
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      b[e] = (k0 + e < k) ? static_cast<uint64_t>(__double_as_longlong(rowp[k0 + e])) : 0ull;
  }
}

// A' + off (mod 2^64) for the fp64 pattern `bits` of an element of a row
// whose largest magnitude is a normal number (or non-finite), with p <= 52:
// |x 2^s| is then a right shift of the 53-bit significand M by
// d = (d0 = 1075 - s) - max(E, 1) >= 1, rounded half to even as
// (M + 2^(d-1) - 1 + bit_d(M)) >> d; d is capped at 54, where every M < 2^53
// gives 0.  Non-finite elements give an unspecified value (they set the
// non-finite flag elsewhere).
__device__ __forceinline__ uint64_t offset_integer_fast(uint64_t bits, int d0, uint64_t off) {
  const uint32_t hi = static_cast<uint32_t>(bits >> 32), lo = static_cast<uint32_t>(bits);
  const uint32_t ah = hi & 0x7FFFFFFFu;
  const uint32_t e20 = max(ah & 0x7FF00000u, 0x00100000u);  // max(E, 1) << 20
  const uint32_t mhi = ah + 0x00100000u - e20;              // M's high word: implicit bit for normals
  const int d = min(d0 - static_cast<int>(e20 >> 20), 54);
  const uint64_t M = (static_cast<uint64_t>(mhi) << 32) | lo;
  const uint64_t q = (M + ((1ull << (d - 1)) - 1ull) + ((M >> d) & 1ull)) >> d;
  const uint64_t neg = static_cast<uint64_t>(static_cast<long long>(static_cast<int>(hi) >> 31));  // 0 or ~0
  return off + ((q ^ neg) - neg);
}

}  // namespace ozemu
