// Per-output reconstruction: residues -> C' by the CRT in direct form
// (integer dot products with the CRT basis and one quotient estimate) ->
// one correct rounding of C' 2^-(s_i + t_j) to fp64.
//
// [TME4] abstract: the per-output reconstruction term of the TME model.
// [AWE] abstract: the residue number system of Ozaki scheme II.
//
// The mixed-radix form (used where the direct form's quotient estimate is
// ambiguous) and the rounding live in crt_device.cuh.
#include <cstdint>

#include "common.cuh"
#include "crt_device.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kCrtThreads = 128;
// Four resident CTAs per SM: at most 128 registers a thread, enough for the
// four outputs' interleaved common paths without spilling.
constexpr int kCrtMinBlocks = 4;

__device__ __forceinline__ uint32_t dp2a_lo(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp2a.lo.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t dp2a_hi(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp2a.hi.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One thread per 4 consecutive outputs of a row.  For each output the
// residues c_l (bytes of four moduli per word) are dotted with the 16-bit
// limbs of the constants W_l = (M/m_l) ((M/m_l)^-1 mod m_l) by two-way dot
// products (dp2a: two 16-bit limbs times two residue bytes; a last single
// modulus by 32-bit multiply-adds):
//   T_t = sum_l c_l limb16_t(W_l) < 2^29,   Y = sum_t T_t 2^(16 t) = sum_l c_l W_l < 2^12 M,
// q = round(Y / M) is estimated in fp32 from the three top T_t (error below
// 2^-9.5), and C' = Y - q M is carried once into 16-bit limbs modulo
// 2^(16 NX) (|C'| < M/2 fits).  When Y/M lies within 2^-8 of a half-integer
// the estimate may be off by one: that output takes the mixed-radix digits
// instead (crt_round), which are exact for any input.
// NLimb = 2: the two-limb moduli (kModulusTable2), whose products have the
// bit lengths kCrtBits2; NLimb = 1: the mixed-digit moduli (kCrtBitsMix).
// Work item g (< 2^31) is output group g % gpr of row g / gpr (gpr = groups
// of four per row), the quotient taken as the high word of g * gdiv with
// gdiv = floor((2^64 - 1) / gpr) + 1 (exact for g, gpr < 2^32).
template <int R, int NLimb>
__global__ void __launch_bounds__(kCrtThreads, kCrtMinBlocks) crt_kernel(int m, int n, const uint8_t* __restrict__ res,
                                                          long long ldr, long long plane,
                                                          const int32_t* __restrict__ sa,
                                                          const int32_t* __restrict__ sb, double* __restrict__ C,
                                                          long long ldc, uint64_t gdiv,
                                                          const __grid_constant__ CrtModuli cm) {
  constexpr bool kLastByMad = (R % 4) == 1;   // a lone last modulus: multiply-adds, not dp2a
  constexpr int NQ = kLastByMad ? R / 4 : (R + 3) / 4;  // words of four residues through dp2a
  constexpr int BM = NLimb == 1 ? kCrtBitsMix[R] : (NLimb == 2 ? kCrtBits2[R] : kCrtBits[R]);  // bit length of M
  constexpr int NT = (BM + 15) / 16;          // 16-bit positions of Y's partial sums
  constexpr int NX = (BM + 15) / 16;          // 16-bit limbs of C' (two's complement)
  static_assert(NX <= 8 && NX <= NT, "C' fits 128 bits");
  const uint32_t gpr = static_cast<uint32_t>((n + 3) / 4);
  const uint32_t total = static_cast<uint32_t>(m) * gpr;
  for (uint32_t g = blockIdx.x * kCrtThreads + threadIdx.x; g < total; g += gridDim.x * kCrtThreads) {
    const uint32_t i = gpr == 1 ? g : static_cast<uint32_t>(__umul64hi(static_cast<uint64_t>(g), gdiv));
    const int j0 = static_cast<int>(g - i * gpr) * 4;
    constexpr int NW = 4 * ((R + 3) / 4);
    uint32_t word[NW];
    const uint8_t* base = res + static_cast<long long>(i) * ldr + j0;
#pragma unroll
    for (int l = 0; l < NW; ++l)
      word[l] = l < R ? __ldcs(reinterpret_cast<const uint32_t*>(base + l * plane)) : 0u;
    // cw[e][q]: residues of moduli 4q .. 4q+3 of output j0 + e.
    uint32_t cw[4][NQ > 0 ? NQ : 1];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      const uint32_t t0 = __byte_perm(word[4 * q], word[4 * q + 1], 0x5140);
      const uint32_t t1 = __byte_perm(word[4 * q + 2], word[4 * q + 3], 0x5140);
      const uint32_t t2 = __byte_perm(word[4 * q], word[4 * q + 1], 0x7362);
      const uint32_t t3 = __byte_perm(word[4 * q + 2], word[4 * q + 3], 0x7362);
      cw[0][q] = __byte_perm(t0, t1, 0x5410);
      cw[1][q] = __byte_perm(t0, t1, 0x7632);
      cw[2][q] = __byte_perm(t2, t3, 0x5410);
      cw[3][q] = __byte_perm(t2, t3, 0x7632);
    }
    const int si = sa[i];
    double* crow = C + static_cast<long long>(i) * ldc + j0;
    // The four outputs' common paths side by side (no branch between them),
    // then the rare ones again by the mixed-radix digits: an ambiguous
    // quotient estimate, or a result in the subnormal range.
    uint64_t bits[4];
    uint32_t rare = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t T[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        uint32_t acc = 0;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          acc = dp2a_lo(cm.w16[q][t][0], cw[e][q], acc);
          if (4 * q + 2 < R) acc = dp2a_hi(cm.w16[q][t][1], cw[e][q], acc);
        }
        if (kLastByMad) {
          const uint32_t c_last = (word[R - 1] >> (8 * e)) & 0xFFu;
          acc += c_last * cm.wl16[t];
        }
        T[t] = acc;
      }
      // q = round(Y / M) from the three top partial sums.
      float yf = 0.f;
#pragma unroll
      for (int t = NT - 3 < 0 ? 0 : NT - 3; t < NT; ++t) yf = fmaf(static_cast<float>(T[t]), cm.gt[t], yf);
      const float qf = rintf(yf);
      if (!(fabsf(yf - qf) < 0.5f - 1.0f / 256.0f)) rare |= 1u << e;
      const int q = static_cast<int>(qf);
      // C' = Y - q M modulo 2^(16 NX), two's complement 16-bit limbs.
      uint32_t x[NX];
      int cr = 0;
#pragma unroll
      for (int t = 0; t < NX; ++t) {
        const int v = static_cast<int>(T[t]) - q * static_cast<int>(cm.m16[t]) + cr;
        x[t] = static_cast<uint32_t>(v) & 0xFFFFu;
        cr = v >> 16;
      }
      uint32_t wds[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint32_t lo = 2 * w < NX ? x[2 * w] : 0u;
        const uint32_t hi = 2 * w + 1 < NX ? x[2 * w + 1] : 0u;
        wds[w] = __byte_perm(lo, hi, 0x5410);
      }
      i128 X = (static_cast<i128>(wds[3]) << 96) | (static_cast<i128>(wds[2]) << 64) |
               (static_cast<i128>(wds[1]) << 32) | static_cast<i128>(wds[0]);
      X = (X << (128 - 16 * NX)) >> (128 - 16 * NX);  // sign-extend from bit 16 NX - 1
      const int S = si + sb[j0 + e < n ? j0 + e : j0];
      bool sub = false;
      bits[e] = round_scaled_normal(X, S, sub);
      if (sub) rare |= 1u << e;
    }
    if (rare) {  // mixed-radix digits, exact for any input, and the general rounding
#pragma unroll 1
      for (int e = 0; e < 4; ++e) {
        if ((rare & (1u << e)) && j0 + e < n) {
          uint32_t c[R];
#pragma unroll
          for (int l = 0; l < R; ++l) c[l] = (word[l] >> (8 * e)) & 0xFFu;
          bits[e] = crt_round<R>(c, si + sb[j0 + e], cm);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (j0 + e < n) crow[e] = __longlong_as_double(static_cast<long long>(bits[e]));
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

template <int R, int NL>
cudaError_t launch_crt_r(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa, const int32_t* sb,
                         double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream) {
  if (cm.r != R) return cudaErrorInvalidValue;
  if (m <= 0 || n <= 0) return cudaSuccess;
  // Row blocks of fewer than 2^31 work items each (the kernel's 32-bit index).
  const long long gpr = (n + 3) / 4;
  const long long rows_per = ((1ll << 31) - 1) / gpr;
  const uint64_t gdiv = ~0ull / static_cast<uint64_t>(gpr) + 1ull;
  const long long plane = static_cast<long long>(m) * ldr;
  for (long long r0 = 0; r0 < m; r0 += rows_per) {
    const int mb = static_cast<int>(m - r0 < rows_per ? m - r0 : rows_per);
    crt_kernel<R, NL><<<grid_for(static_cast<long long>(mb) * gpr, kCrtThreads), kCrtThreads, 0, stream>>>(
        mb, n, residues + r0 * ldr, ldr, plane, sa + r0, sb, C + r0 * ldc, ldc, gdiv, cm);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_crt_f64(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa,
                           const int32_t* sb, double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream) {
  if (cm.limbs == 1) {  // mixed-digit moduli: r up to kMaxModuliMix
    switch (cm.r) {
#define OZEMU_CRT_MIX(R) \
  case R:                \
    return launch_crt_r<R, 1>(m, n, residues, ldr, sa, sb, C, ldc, cm, stream);
      OZEMU_CRT_MIX(1) OZEMU_CRT_MIX(2) OZEMU_CRT_MIX(3) OZEMU_CRT_MIX(4) OZEMU_CRT_MIX(5) OZEMU_CRT_MIX(6)
      OZEMU_CRT_MIX(7) OZEMU_CRT_MIX(8) OZEMU_CRT_MIX(9) OZEMU_CRT_MIX(10) OZEMU_CRT_MIX(11) OZEMU_CRT_MIX(12)
      OZEMU_CRT_MIX(13) OZEMU_CRT_MIX(14) OZEMU_CRT_MIX(15) OZEMU_CRT_MIX(16) OZEMU_CRT_MIX(17)
      OZEMU_CRT_MIX(18) OZEMU_CRT_MIX(19) OZEMU_CRT_MIX(20)
#undef OZEMU_CRT_MIX
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (cm.r) {
#define OZEMU_CRT_CASE(R) \
  case R:                 \
    return cm.limbs == 2 ? launch_crt_r<R, 2>(m, n, residues, ldr, sa, sb, C, ldc, cm, stream) \
                         : launch_crt_r<R, 3>(m, n, residues, ldr, sa, sb, C, ldc, cm, stream);
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
