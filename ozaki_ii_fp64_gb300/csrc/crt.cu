// Per-output reconstruction: residues -> C' by mixed-radix (Garner) CRT ->
// one correct rounding of C' 2^-(s_i + t_j) to fp64.
//
// [TME4] abstract: the per-output reconstruction term of the TME model.
// [AWE] abstract: the residue number system of Ozaki scheme II.
//
// Balanced mixed-radix digits v_l in [-floor(m_l/2), ceil(m_l/2) - 1] give
// X = sum_l v_l (m_0 ... m_{l-1}) in [-M/2, M/2 - 1] (m_0 = 256 even, the
// rest odd), which is the symmetric representative C' directly.  The digit
// recurrence is v_l = c_l inv_l - sum_{j<l} v_j g_{l,j} (mod m_l), with
// inv_l = (m_0...m_{l-1})^-1 and g_{l,j} = (m_0...m_{j-1}) inv_l mod m_l.
// X is evaluated by Horner's rule on 32-bit words; the conversion to fp64 rounds to
// nearest-even once, including the subnormal range and overflow to inf.
// No fp64 arithmetic is used.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

typedef unsigned __int128 u128;
typedef __int128 i128;

__device__ __forceinline__ int clz128(u128 x) {
  uint64_t hi = static_cast<uint64_t>(x >> 64), lo = static_cast<uint64_t>(x);
  return hi ? __clzll(static_cast<long long>(hi)) : 64 + __clzll(static_cast<long long>(lo));
}

// Bits of RN(X 2^-S) as an IEEE binary64.
__device__ uint64_t round_scaled(i128 X, int S) {
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

constexpr int kCrtThreads = 128;

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

template <int R>
__global__ void __launch_bounds__(kCrtThreads) crt_kernel(int m, int n, const uint8_t* __restrict__ res,
                                                          long long ldr, const int32_t* __restrict__ sa,
                                                          const int32_t* __restrict__ sb, double* __restrict__ C,
                                                          long long ldc, const CrtModuli cm) {
  constexpr int L = Limbs<R>::value;
  const long long groups_per_row = (n + 3) / 4;
  const long long total = static_cast<long long>(m) * groups_per_row;
  const long long plane = static_cast<long long>(m) * ldr;
  for (long long g = blockIdx.x * static_cast<long long>(kCrtThreads) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * kCrtThreads) {
    const int i = static_cast<int>(g / groups_per_row);
    const int j0 = static_cast<int>(g % groups_per_row) * 4;
    uint32_t word[R];
    const uint8_t* base = res + static_cast<long long>(i) * ldr + j0;
#pragma unroll
    for (int l = 0; l < R; ++l) word[l] = __ldcs(reinterpret_cast<const uint32_t*>(base + l * plane));
    const int si = sa[i];
#pragma unroll 1
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      if (j >= n) break;
      // Balanced mixed-radix digits.
      int v[R];
#pragma unroll
      for (int l = 0; l < R; ++l) {
        const uint32_t c = (word[l] >> (8 * e)) & 0xFFu;
        int t = static_cast<int>(c * cm.inv[l]);
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
      const uint64_t bits = round_scaled(X, si + sb[j]);
      C[static_cast<long long>(i) * ldc + j] = __longlong_as_double(static_cast<long long>(bits));
    }
  }
}

template <typename T>
__global__ void zero_kernel(T* C, int m, int n, long long ldc) {
  const long long total = static_cast<long long>(m) * n;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<long long>(gridDim.x) * blockDim.x)
    C[(idx / n) * ldc + idx % n] = T(0);
}

int grid_for(long long work, int threads) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long g = (work + threads - 1) / threads;
  long long cap = static_cast<long long>(sms) * 16;
  return static_cast<int>(g < cap ? (g < 1 ? 1 : g) : cap);
}

}  // namespace

template <int R>
cudaError_t launch_crt_r(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa, const int32_t* sb,
                         double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream) {
  const long long work = static_cast<long long>(m) * ((n + 3) / 4);
  crt_kernel<R><<<grid_for(work, kCrtThreads), kCrtThreads, 0, stream>>>(m, n, residues, ldr, sa, sb, C, ldc, cm);
  return cudaGetLastError();
}

cudaError_t launch_crt_f64(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa,
                           const int32_t* sb, double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream) {
  switch (cm.r) {
#define OZEMU_CRT_CASE(R) \
  case R:                 \
    return launch_crt_r<R>(m, n, residues, ldr, sa, sb, C, ldc, cm, stream);
    OZEMU_CRT_CASE(1) OZEMU_CRT_CASE(2) OZEMU_CRT_CASE(3) OZEMU_CRT_CASE(4) OZEMU_CRT_CASE(5) OZEMU_CRT_CASE(6)
    OZEMU_CRT_CASE(7) OZEMU_CRT_CASE(8) OZEMU_CRT_CASE(9) OZEMU_CRT_CASE(10) OZEMU_CRT_CASE(11)
    OZEMU_CRT_CASE(12) OZEMU_CRT_CASE(13) OZEMU_CRT_CASE(14) OZEMU_CRT_CASE(15) OZEMU_CRT_CASE(16)
#undef OZEMU_CRT_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_zero_f64(double* C, int m, int n, long long ldc, cudaStream_t stream) {
  zero_kernel<double><<<grid_for(static_cast<long long>(m) * n, 256), 256, 0, stream>>>(C, m, n, ldc);
  return cudaGetLastError();
}

cudaError_t launch_zero_s32(int32_t* C, int m, int n, long long ldc, cudaStream_t stream) {
  zero_kernel<int32_t><<<grid_for(static_cast<long long>(m) * n, 256), 256, 0, stream>>>(C, m, n, ldc);
  return cudaGetLastError();
}

}  // namespace ozemu
