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

__device__ __forceinline__ uint32_t dp4a_u8(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// One thread per 4 consecutive outputs of a row.  For each output the
// residues c_l (bytes of four moduli per word) are dotted with the bytes of
// the constants W_l = (M/m_l) ((M/m_l)^-1 mod m_l) by dp4a (a last single
// modulus by 32-bit multiply-adds on 16-bit limbs):
//   T_t = sum_l c_l limb16_t(W_l) < 2^29,   Y = sum_t T_t 2^(16 t) = sum_l c_l W_l < 2^12 M,
// q = round(Y / M) is estimated in fp32 from the three top T_t (error below
// 2^-9.5), and C' = Y - q M is carried once into 16-bit limbs modulo
// 2^(16 NX) (|C'| < M/2 fits).  When Y/M lies within 2^-8 of a half-integer
// the estimate may be off by one: that output takes the mixed-radix digits
// instead (crt_round), which are exact for any input.
// NLimb = 2: the two-limb moduli (kModulusTable2), whose products have the
// bit lengths kCrtBits2; NLimb = 1: the mixed-digit moduli (kCrtBitsMix).
template <int R, int NLimb>
__global__ void __launch_bounds__(kCrtThreads) crt_kernel(int m, int n, const uint8_t* __restrict__ res,
                                                          long long ldr, const int32_t* __restrict__ sa,
                                                          const int32_t* __restrict__ sb, double* __restrict__ C,
                                                          long long ldc, const __grid_constant__ CrtModuli cm) {
  constexpr bool kLastByMad = (R % 4) == 1;   // a lone last modulus: multiply-adds, not dp4a
  constexpr int NQ = kLastByMad ? R / 4 : (R + 3) / 4;  // words of four residues through dp4a
  constexpr int BM = NLimb == 1 ? kCrtBitsMix[R] : (NLimb == 2 ? kCrtBits2[R] : kCrtBits[R]);  // bit length of M
  constexpr int NL = (BM + 7) / 8;            // bytes of W_l
  constexpr int NT = (NL + 1) / 2;            // 16-bit positions of Y's partial sums
  constexpr int NX = (BM + 15) / 16;          // 16-bit limbs of C' (two's complement)
  static_assert(NX <= 8 && NX <= NT, "C' fits 128 bits");
  const long long groups_per_row = (n + 3) / 4;
  const long long total = static_cast<long long>(m) * groups_per_row;
  const long long plane = static_cast<long long>(m) * ldr;
  for (long long g = blockIdx.x * static_cast<long long>(kCrtThreads) + threadIdx.x; g < total;
       g += static_cast<long long>(gridDim.x) * kCrtThreads) {
    const int i = static_cast<int>(g / groups_per_row);
    const int j0 = static_cast<int>(g % groups_per_row) * 4;
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
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = j0 + e;
      if (j >= n) continue;
      uint32_t T[NT];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        uint32_t s0 = 0, s1 = 0;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          s0 = dp4a_u8(cw[e][q], cm.wb[q][2 * t], s0);
          if (2 * t + 1 < NL) s1 = dp4a_u8(cw[e][q], cm.wb[q][2 * t + 1], s1);
        }
        T[t] = s0 + (s1 << 8);
        if (kLastByMad) {
          const uint32_t c_last = (word[R - 1] >> (8 * e)) & 0xFFu;
          T[t] += c_last * cm.wl16[t];
        }
      }
      // q = round(Y / M) from the three top partial sums.
      float yf = 0.f;
#pragma unroll
      for (int t = NT - 3 < 0 ? 0 : NT - 3; t < NT; ++t) yf = fmaf(static_cast<float>(T[t]), cm.gt[t], yf);
      const float qf = rintf(yf);
      const int S = si + sb[j];
      uint64_t bits;
      if (fabsf(yf - qf) < 0.5f - 1.0f / 256.0f) {
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
        bits = round_scaled_fast(X, S);
      } else {
        uint32_t c[R];
#pragma unroll
        for (int l = 0; l < R; ++l) c[l] = (word[l] >> (8 * e)) & 0xFFu;
        bits = crt_round<R>(c, S, cm);
      }
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

template <int R, int NL>
cudaError_t launch_crt_r(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa, const int32_t* sb,
                         double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream) {
  if (cm.r != R) return cudaErrorInvalidValue;
  const long long work = static_cast<long long>(m) * ((n + 3) / 4);
  crt_kernel<R, NL><<<grid_for(work, kCrtThreads), kCrtThreads, 0, stream>>>(m, n, residues, ldr, sa, sb, C, ldc, cm);
  return cudaGetLastError();
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
