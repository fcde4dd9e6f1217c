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
// X is accumulated as a 128-bit integer; the conversion to fp64 rounds to
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

__global__ void __launch_bounds__(kCrtThreads) crt_kernel(int m, int n, const uint8_t* __restrict__ res,
                                                          long long ldr, const int32_t* __restrict__ sa,
                                                          const int32_t* __restrict__ sb, double* __restrict__ C,
                                                          long long ldc, const CrtModuli cm) {
  const long long groups_per_row = (n + 3) / 4;
  const long long total = static_cast<long long>(m) * groups_per_row;
  const int r = cm.r;
  const long long plane = static_cast<long long>(m) * ldr;
  for (long long g = blockIdx.x * static_cast<long long>(kCrtThreads) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * kCrtThreads) {
    const int i = static_cast<int>(g / groups_per_row);
    const int j0 = static_cast<int>(g % groups_per_row) * 4;
    uint32_t word[kMaxModuli];
    const uint8_t* base = res + static_cast<long long>(i) * ldr + j0;
#pragma unroll
    for (int l = 0; l < kMaxModuli; ++l)
      word[l] = (l < r) ? __ldcs(reinterpret_cast<const uint32_t*>(base + l * plane)) : 0u;
    const int si = sa[i];
#pragma unroll 1
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      if (j >= n) break;
      int v[kMaxModuli];
      i128 X = 0;
#pragma unroll
      for (int l = 0; l < kMaxModuli; ++l) {
        if (l < r) {
          const uint32_t c = (word[l] >> (8 * e)) & 0xFFu;
          int t = static_cast<int>(c * cm.inv[l]);
#pragma unroll
          for (int jj = 0; jj < l; ++jj) t -= v[jj] * static_cast<int>(cm.g[l][jj]);
          const uint32_t ml = cm.m[l];
          uint32_t tp = static_cast<uint32_t>(t + static_cast<int>(ml << 13));
          uint32_t q = __umulhi(tp, cm.magic[l]);
          uint32_t rr = tp - q * ml;
          rr = rr >= ml ? rr - ml : rr;
          v[l] = static_cast<int>(rr) - (rr > (ml - 1) / 2 ? static_cast<int>(ml) : 0);
          const u128 pref = (static_cast<u128>(cm.prefix[l][3]) << 96) | (static_cast<u128>(cm.prefix[l][2]) << 64) |
                            (static_cast<u128>(cm.prefix[l][1]) << 32) | static_cast<u128>(cm.prefix[l][0]);
          X += static_cast<i128>(v[l]) * static_cast<i128>(pref);
        }
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

cudaError_t launch_crt_f64(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa,
                           const int32_t* sb, double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream) {
  const long long work = static_cast<long long>(m) * ((n + 3) / 4);
  crt_kernel<<<grid_for(work, kCrtThreads), kCrtThreads, 0, stream>>>(m, n, residues, ldr, sa, sb, C, ldc, cm);
  return cudaGetLastError();
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
