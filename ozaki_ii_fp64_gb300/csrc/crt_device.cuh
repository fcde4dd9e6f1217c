// Device-side CRT and scale back shared by the CRT kernel and the fused
// narrow-N kernel: residues c_l in [0, m_l) -> balanced mixed-radix (Garner)
// digits -> C' on 32-bit words -> one correct rounding of C' 2^-S to fp64.
//
// [AWE] abstract: the residue number system of Ozaki scheme II.
// [TME4] abstract: the per-output reconstruction term.
//
// Balanced digits v_l in [-floor(m_l/2), ceil(m_l/2) - 1] give
// X = sum_l v_l (m_0 ... m_{l-1}) = C' (mod M).  When the one even modulus
// comes first (256; 8 for the mixed-digit moduli; the other moduli odd), X
// lies in [-M/2, M/2 - 1] and is the symmetric representative C' directly;
// with the even modulus elsewhere (112, second of the two-limb moduli) X can
// lie up to m_0/2 outside it, so X is brought into [-M/2, M/2) by +-M.  The digit
// recurrence is v_l = c_l inv_l - sum_{j<l} v_j g_{l,j} (mod m_l), with
// inv_l = (m_0...m_{l-1})^-1 and g_{l,j} = (m_0...m_{j-1}) inv_l mod m_l.
// No fp64 arithmetic is used.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace ozemu {

typedef unsigned __int128 u128;
typedef __int128 i128;

__device__ __forceinline__ int clz128(u128 x) {
  uint64_t hi = static_cast<uint64_t>(x >> 64), lo = static_cast<uint64_t>(x);
  return hi ? __clzll(static_cast<long long>(hi)) : 64 + __clzll(static_cast<long long>(lo));
}

// Bits of RN(X 2^-S) as an IEEE binary64 (the rare subnormal-range path:
// not inlined, so it does not widen the common path).
__device__ __noinline__ uint64_t round_scaled(i128 X, int S) {
  if (X == 0) return 0ull;
  const bool neg = X < 0;
  u128 mag = neg ? static_cast<u128>(-X) : static_cast<u128>(X);
  const int b = 127 - clz128(mag);           // top bit index
  int sh = b - 52;                           // keep 53 significant bits ...
  if (S - 1074 > sh) sh = S - 1074;          // ... or fewer in the subnormal range
  uint64_t q;
  if (sh <= 0) {
    q = static_cast<uint64_t>(mag << (-sh));
  } else if (sh >= 128) {
    q = 0;  // |X| < 2^126 <= 2^(sh-1): rounds to zero
  } else {
    u128 qq = mag >> sh;
    u128 rem = mag - (qq << sh);
    u128 half = static_cast<u128>(1) << (sh - 1);
    q = static_cast<uint64_t>(qq);
    if (rem > half || (rem == half && (q & 1ull))) ++q;
  }
  if (q >> 53) {  // rounding carried into bit 53: q == 2^53
    q >>= 1;
    ++sh;
  }
  uint64_t bits;
  if (q < (1ull << 52)) {
    bits = q;  // subnormal (or zero)
  } else {
    const long long E = static_cast<long long>(sh) - S + 52 + 1023;
    if (E >= 2047)
      bits = 0x7FF0000000000000ull;
    else
      bits = (static_cast<uint64_t>(E) << 52) | (q & 0xFFFFFFFFFFFFFull);
  }
  return neg ? (bits | 0x8000000000000000ull) : bits;
}

// round_scaled for a normal (or overflowing) result, on the words of X: the
// top 64 bits of |X| and a sticky bit.  A result in the subnormal range sets
// sub and returns an unspecified value (round_scaled takes it).
__device__ __forceinline__ uint64_t round_scaled_normal(i128 X, int S, bool& sub) {
  sub = false;
  if (X == 0) return 0ull;
  const bool neg = X < 0;
  const u128 mag = neg ? static_cast<u128>(-X) : static_cast<u128>(X);
  const uint64_t hi = static_cast<uint64_t>(mag >> 64), lo = static_cast<uint64_t>(mag);
  uint64_t M;
  bool sticky;
  int e;  // index of the leading bit of |X|
  if (hi != 0) {
    const int lz = __clzll(static_cast<long long>(hi));
    M = lz ? (hi << lz) | (lo >> (64 - lz)) : hi;
    sticky = lz ? (lo << lz) != 0 : lo != 0;
    e = 127 - lz;
  } else {
    const int lz = __clzll(static_cast<long long>(lo));
    M = lo << lz;
    sticky = false;
    e = 63 - lz;
  }
  int b = e - S;  // exponent of the result's leading bit
  sub = b < -1022;
  uint64_t q = M >> 11;
  const uint64_t rb = (M >> 10) & 1ull;
  const bool st = sticky || (M & 0x3FFull) != 0;
  q += rb & static_cast<uint64_t>(st | (q & 1ull));
  if (q >> 53) {
    q >>= 1;
    ++b;
  }
  const uint64_t bits =
      b > 1023 ? 0x7FF0000000000000ull : (static_cast<uint64_t>(b + 1023) << 52) | (q & 0xFFFFFFFFFFFFFull);
  return neg ? (bits | 0x8000000000000000ull) : bits;
}

// Number of 32-bit words that hold +-M/2 for the first R moduli (M < 2^(8R),
// and M < 2^126 for every R <= 16, so four words always suffice).
template <int R>
struct Limbs {
  static constexpr int value = (8 * R + 1 + 31) / 32 < 4 ? (8 * R + 1 + 31) / 32 : 4;
};

// X <- X * m + v on a two's-complement integer of L 32-bit words (v signed,
// |v| <= 128, m <= 256; no overflow because |X * m + v| < M/2 throughout).
template <int L>
__device__ __forceinline__ void horner_step(uint32_t (&x)[L], uint32_t m, int v) {
  const uint32_t sx = v < 0 ? 0xFFFFFFFFu : 0u;
  uint64_t t = static_cast<uint64_t>(x[0]) * m + static_cast<uint32_t>(v);
  x[0] = static_cast<uint32_t>(t);
#pragma unroll
  for (int w = 1; w < L; ++w) {
    t = static_cast<uint64_t>(x[w]) * m + (t >> 32) + sx;
    x[w] = static_cast<uint32_t>(t);
  }
}

// Bits of RN(C' 2^-S) for the residues c[0..R) (each in [0, m_l)); the
// CRT kernel's fallback, not inlined.
template <int R>
__device__ __noinline__ uint64_t crt_round(const uint32_t (&c)[R], int S, const CrtModuli& cm) {
  constexpr int L = Limbs<R>::value;
  int v[R];
#pragma unroll
  for (int l = 0; l < R; ++l) {
    int t = static_cast<int>(c[l] * cm.inv[l]);
#pragma unroll
    for (int jj = 0; jj < l; ++jj) t -= v[jj] * static_cast<int>(cm.g[l][jj]);
    const uint32_t ml = cm.m[l];
    const uint32_t tp = static_cast<uint32_t>(t + static_cast<int>(ml << 13));  // > 0, < 2^22
    const uint32_t q = __umulhi(tp, cm.magic[l]);
    uint32_t rr = tp - q * ml;
    rr = rr >= ml ? rr - ml : rr;
    v[l] = static_cast<int>(rr) - (rr > (ml - 1) / 2 ? static_cast<int>(ml) : 0);
  }
  // X = v_0 + m_0 (v_1 + m_1 (v_2 + ...)), Horner from the top digit.
  uint32_t x[L];
  const uint32_t top_sign = v[R - 1] < 0 ? 0xFFFFFFFFu : 0u;
  x[0] = static_cast<uint32_t>(v[R - 1]);
#pragma unroll
  for (int w = 1; w < L; ++w) x[w] = top_sign;
#pragma unroll
  for (int l = R - 2; l >= 0; --l) horner_step<L>(x, cm.m[l], v[l]);
  i128 X = 0;
#pragma unroll
  for (int w = L - 1; w >= 0; --w) X = (X << 32) | static_cast<i128>(x[w]);
  if (L < 4) {  // sign-extend from 32 L bits
    const int sh = 128 - 32 * L;
    X = (X << sh) >> sh;
  }
  i128 M = 0;
#pragma unroll
  for (int t = 7; t >= 0; --t) M = (M << 16) | static_cast<i128>(cm.m16[t]);
  if (2 * X >= M) X -= M;
  else if (2 * X < -M) X += M;
  return round_scaled(X, S);
}

}  // namespace ozemu
