// Per-output reconstruction: residues -> C' by mixed-radix (Garner) CRT ->
// one correct rounding of C' 2^-(s_i + t_j) to fp64.
//
// [TME4] abstract: the per-output reconstruction term of the TME model.
// [AWE] abstract: the residue number system of Ozaki scheme II.
//
// The digit recurrence, Horner evaluation and rounding live in
// crt_device.cuh.
#include <cstdint>

#include "common.cuh"
#include "crt_device.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kCrtThreads = 128;

template <int R>
__global__ void __launch_bounds__(kCrtThreads) crt_kernel(int m, int n, const uint8_t* __restrict__ res,
                                                          long long ldr, const int32_t* __restrict__ sa,
                                                          const int32_t* __restrict__ sb, double* __restrict__ C,
                                                          long long ldc, const CrtModuli cm) {
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
      uint32_t c[R];
#pragma unroll
      for (int l = 0; l < R; ++l) c[l] = (word[l] >> (8 * e)) & 0xFFu;
      const uint64_t bits = crt_round<R>(c, si + sb[j], cm);
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
