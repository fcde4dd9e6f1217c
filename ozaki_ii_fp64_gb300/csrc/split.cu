// Deconstruction kernels: fp64 rows -> power-of-two scale -> integer ->
// balanced residues modulo r moduli -> base-13 FP4 limb planes; int8 rows ->
// limb planes; and the transposes used for column splits.
//
// Follows [TME4] abstract (every streamed fp64 operand is scaled, rounded
// and reduced modulo each of the r moduli on SIMT pipes) and [AWE] abstract
// (residues split with carries into base-13 digits from S, stored as FP4).
//
// All fp64 handling is integer bit manipulation: no fp64 arithmetic.
#include <cstdint>

#include "common.cuh"
#include "deconstruct.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kSplitThreads = 256;
constexpr int kElemsPerThread = 8;
constexpr int kChunk = kSplitThreads * kElemsPerThread;  // elements of a row per pass step
constexpr int kLutStride = 512;                          // u32 entries per modulus (>= 2 m)

// Smallest-magnitude member of S = {0,+-1,+-2,+-3,+-4,+-6,+-8,+-12} in the
// class c mod 13 (c in [0, 13)).  Classes 1 and 12 take 1 and -1.
__device__ int class_digit(int c) {
  switch (c) {
    case 5: return -8;
    case 7: return -6;
    case 9: return -4;
    case 10: return -3;
    case 11: return -2;
    case 12: return -1;
    default: return c;  // 0, 1, 2, 3, 4, 6, 8
  }
}

// 4-bit e2m1 code of the FP4 value d/2 for d in S.
__device__ uint32_t e2m1_nibble(int d) {
  int a = d < 0 ? -d : d;
  uint32_t mag = (a <= 4) ? static_cast<uint32_t>(a) : (a == 6 ? 5u : (a == 8 ? 6u : 7u));
  return (d < 0 ? 8u : 0u) | mag;
}

__device__ int mod13(int x) {
  int c = x % 13;
  return c < 0 ? c + 13 : c;
}

// Limb codes of an integer x in [-128, 127]: three nibbles in bytes 0, 1, 2.
__device__ uint32_t limb_code(int x) {
  int d0 = class_digit(mod13(x));
  x = (x - d0) / 13;
  int d1 = class_digit(mod13(x));
  int d2 = (x - d1) / 13;  // in {-1, 0, 1} for int8 inputs
  return e2m1_nibble(d0) | (e2m1_nibble(d1) << 8) | (e2m1_nibble(d2) << 16);
}

// Packs 8 limb codes (nibbles in bytes 0..2) into the three plane words:
// word j holds limb j of elements 0..7, element e in nibble e.
__device__ __forceinline__ void pack8(const uint32_t (&c)[8], uint32_t& w0, uint32_t& w1, uint32_t& w2) {
  uint32_t p01 = c[0] | (c[1] << 4);
  uint32_t p23 = c[2] | (c[3] << 4);
  uint32_t p45 = c[4] | (c[5] << 4);
  uint32_t p67 = c[6] | (c[7] << 4);
  uint32_t lo = __byte_perm(p01, p23, 0x5140);
  uint32_t hi = __byte_perm(p45, p67, 0x5140);
  w0 = __byte_perm(lo, hi, 0x5410);
  w1 = __byte_perm(lo, hi, 0x7632);
  uint32_t ulo = __byte_perm(p01, p23, 0x0062);
  uint32_t uhi = __byte_perm(p45, p67, 0x0062);
  w2 = __byte_perm(ulo, uhi, 0x5410);
}

// Pass 2 of the row split over the row's elements: integers, residues and
// limb codes (or residue bytes), packed and stored.
template <int R, bool kRes8, bool kFast>
__device__ __forceinline__ void split_pass2(const double* rowp, int k, int k_p, int vec_ok, int s,
                                            const SplitModuli& mods, const uint32_t* lut, uint8_t* out_row,
                                            long long plane_stride) {
  for (int k0 = threadIdx.x * kElemsPerThread; k0 < k_p; k0 += kChunk) {
    uint64_t b[8];
    load8_f64(rowp, k, k0, vec_ok, b, true);
    uint32_t a2[8], a1[8], a0x4[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint64_t u = kFast ? offset_integer_fast(b[e], 1075 - s, 1ull << 62) : scaled_offset(b[e], s);
      a0x4[e] = (static_cast<uint32_t>(u) & 0x1FFFFFu) << 2;
      a1[e] = static_cast<uint32_t>(u >> 21) & 0x1FFFFFu;
      a2[e] = static_cast<uint32_t>(u >> 42);
    }
    uint32_t* o = reinterpret_cast<uint32_t*>(out_row + (kRes8 ? k0 : k0 / 2));
#pragma unroll
    for (int l = 0; l < R; ++l) {
      const uint32_t c21 = mods.c21x4[l], c42 = mods.c42x4[l], mg = mods.magic4[l], m4 = mods.m[l] * 4u;
      const char* lt = reinterpret_cast<const char*>(lut + l * kLutStride);
      uint32_t c[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint32_t v4 = a2[e] * c42 + (a1[e] * c21 + a0x4[e]);
        uint32_t q = __umulhi(v4, mg);
        uint32_t off = v4 - q * m4;
        c[e] = *reinterpret_cast<const uint32_t*>(lt + off);
      }
      if constexpr (kRes8) {
        uint2 w;
        w.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
        w.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
        __stcs(reinterpret_cast<uint2*>(o + static_cast<long long>(l) * plane_stride / 4), w);
      } else {
        uint32_t w0, w1, w2;
        pack8(c, w0, w1, w2);
        const long long pl = static_cast<long long>(l * 3) * plane_stride / 4;
        __stcs(o + pl, w0);
        __stcs(o + pl + plane_stride / 4, w1);
        __stcs(o + pl + 2 * plane_stride / 4, w2);
      }
    }
  }
}

// kRes8 = false: FP4 limb planes [r][3][rows_p][k_p/2] (the FP4 path).
// kRes8 = true: the balanced residues themselves as int8 [r][rows_p][k_p]
// (input of the INT8 comparison GEMM).
template <int R, bool kRes8>
__global__ void __launch_bounds__(kSplitThreads, 3)
    split_rows_f64_kernel(const double* __restrict__ X, long long ldx, int rows, int k, int rows_p, int k_p, int p,
                          SplitModuli mods, uint8_t* __restrict__ planes, int32_t* __restrict__ shifts,
                          uint32_t* flags) {
  extern __shared__ __align__(16) uint32_t lut[];  // [R][kLutStride]
  __shared__ uint64_t red[kSplitThreads / 32];
  constexpr int r = R;
  for (int l = 0; l < r; ++l) {
    const uint32_t m = mods.m[l];
    for (uint32_t i = threadIdx.x; i < 2 * m; i += kSplitThreads) {
      uint32_t res = (i + m - mods.off[l]) % m;  // residue of x' = u - 2^62
      int bal = static_cast<int>(res) - (res > (m - 1) / 2 ? static_cast<int>(m) : 0);
      lut[l * kLutStride + i] = kRes8 ? static_cast<uint32_t>(static_cast<uint8_t>(bal)) : limb_code(bal);
    }
  }
  __syncthreads();

  const long long row_bytes = kRes8 ? k_p : k_p / 2;
  const long long plane_stride = static_cast<long long>(rows_p) * row_bytes;
  constexpr int kPlanesPerModulus = kRes8 ? 1 : 3;
  const int vec_ok = row_vector_width(X, ldx);

  for (int row = blockIdx.x; row < rows_p; row += gridDim.x) {
    uint8_t* out_row = planes + static_cast<long long>(row) * row_bytes;
    if (row >= rows) {  // padding row: digit (or residue) 0 everywhere
      for (int l = 0; l < r; ++l)
        for (int j = 0; j < kPlanesPerModulus; ++j) {
          uint32_t* o = reinterpret_cast<uint32_t*>(out_row + (l * kPlanesPerModulus + j) * plane_stride);
          for (int w = threadIdx.x; w < row_bytes / 4; w += kSplitThreads) o[w] = 0u;
        }
      continue;
    }
    const double* rowp = X + static_cast<long long>(row) * ldx;

    // Pass 1: largest magnitude of the row (as an ordered bit pattern).
    uint64_t mx = 0;
    for (int k0 = threadIdx.x * kElemsPerThread; k0 < k; k0 += kChunk) {
      uint64_t b[8];
      load8_f64(rowp, k, k0, vec_ok, b, false);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        uint64_t a = b[e] & 0x7FFFFFFFFFFFFFFFull;
        mx = a > mx ? a : mx;
      }
    }
    mx = block_max_u64<kSplitThreads>(mx, red);
    int s = 0;
    if (mx != 0) s = p - frexp_exp_bits(mx);
    if (mx >= 0x7FF0000000000000ull && threadIdx.x == 0) atomicOr(flags, kFlagNonFinite);
    if (threadIdx.x == 0) shifts[row] = s;

    // Pass 2: integers, residues, limbs.  Rows whose largest magnitude is
    // normal (with p <= 52) take the right-shift rounding.
    if ((mx >> 52) != 0 && p <= 52)
      split_pass2<R, kRes8, true>(rowp, k, k_p, vec_ok, s, mods, lut, out_row, plane_stride);
    else
      split_pass2<R, kRes8, false>(rowp, k, k_p, vec_ok, s, mods, lut, out_row, plane_stride);
  }
}

__global__ void __launch_bounds__(kSplitThreads) split_rows_s8_kernel(const int8_t* __restrict__ X, long long ldx,
                                                                     int rows, int k, int rows_p, int k_p,
                                                                     uint8_t* __restrict__ planes) {
  __shared__ uint32_t lut[256];
  for (int i = threadIdx.x; i < 256; i += kSplitThreads) lut[i] = limb_code(i - 128);
  __syncthreads();
  const long long row_bytes = k_p / 2;
  const long long plane_words = static_cast<long long>(rows_p) * row_bytes / 4;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(X) & 7u) == 0) && ((ldx & 7) == 0);
  for (int row = blockIdx.x; row < rows_p; row += gridDim.x) {
    uint32_t* o_row = reinterpret_cast<uint32_t*>(planes + static_cast<long long>(row) * row_bytes);
    const int8_t* rowp = X + static_cast<long long>(row) * ldx;
    for (int k0 = threadIdx.x * kElemsPerThread; k0 < k_p; k0 += kChunk) {
      int8_t v[8];
      if (row < rows && vec_ok && k0 + 8 <= k) {
        uint2 w = __ldcs(reinterpret_cast<const uint2*>(rowp + k0));
        const int8_t* pv = reinterpret_cast<const int8_t*>(&w);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = pv[e];
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (row < rows && k0 + e < k) ? rowp[k0 + e] : static_cast<int8_t>(0);
      }
      uint32_t c[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = lut[static_cast<int>(v[e]) + 128];
      uint32_t w0, w1, w2;
      pack8(c, w0, w1, w2);
      uint32_t* o = o_row + k0 / 8;
      o[0] = w0;
      o[plane_words] = w1;
      o[2 * plane_words] = w2;
    }
  }
}

// out[c][r] = in[r][c] for a rows x cols block of 32 x 32 tiles.
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ in, long long ldin, int rows, int cols, T* __restrict__ out,
                                 long long ldout) {
  __shared__ T tile[32][33];
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    int rr = r0 + i, cc = c0 + threadIdx.x;
    if (rr < rows && cc < cols) tile[i][threadIdx.x] = in[static_cast<long long>(rr) * ldin + cc];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    int cc = c0 + i, rr = r0 + threadIdx.x;
    if (rr < rows && cc < cols) out[static_cast<long long>(cc) * ldout + rr] = tile[threadIdx.x][i];
  }
}

int split_grid(int rows_p) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int g = sms * 3;  // three CTAs per SM fit (80 registers x 256 threads)
  return rows_p < g ? rows_p : g;
}

}  // namespace

template <int R, bool kRes8>
cudaError_t launch_split_r(const double* X, long long ldx, int rows, int k, int p, const SplitModuli& mods,
                           uint8_t* planes, int32_t* shifts, uint32_t* flags, cudaStream_t stream) {
  const int rows_p = round_up(rows, kRowAlign), k_p = round_up(k, kKAlign);
  const size_t smem = static_cast<size_t>(R) * kLutStride * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(split_rows_f64_kernel<R, kRes8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  split_rows_f64_kernel<R, kRes8><<<split_grid(rows_p), kSplitThreads, smem, stream>>>(X, ldx, rows, k, rows_p, k_p,
                                                                                       p, mods, planes, shifts, flags);
  return cudaGetLastError();
}

template <bool kRes8>
cudaError_t launch_split_mode(const double* X, long long ldx, int rows, int k, int p, const SplitModuli& mods,
                              uint8_t* planes, int32_t* shifts, uint32_t* flags, cudaStream_t stream) {
  switch (mods.r) {
#define OZEMU_SPLIT_CASE(R) \
  case R:                   \
    return launch_split_r<R, kRes8>(X, ldx, rows, k, p, mods, planes, shifts, flags, stream);
    OZEMU_SPLIT_CASE(1) OZEMU_SPLIT_CASE(2) OZEMU_SPLIT_CASE(3) OZEMU_SPLIT_CASE(4) OZEMU_SPLIT_CASE(5)
    OZEMU_SPLIT_CASE(6) OZEMU_SPLIT_CASE(7) OZEMU_SPLIT_CASE(8) OZEMU_SPLIT_CASE(9) OZEMU_SPLIT_CASE(10)
    OZEMU_SPLIT_CASE(11) OZEMU_SPLIT_CASE(12) OZEMU_SPLIT_CASE(13) OZEMU_SPLIT_CASE(14) OZEMU_SPLIT_CASE(15)
    OZEMU_SPLIT_CASE(16)
#undef OZEMU_SPLIT_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_split_rows_f64(const double* X, long long ldx, int rows, int k, int p, const SplitModuli& mods,
                                  uint8_t* planes, int32_t* shifts, uint32_t* flags, cudaStream_t stream) {
  return launch_split_mode<false>(X, ldx, rows, k, p, mods, planes, shifts, flags, stream);
}

cudaError_t launch_split_rows_f64_res8(const double* X, long long ldx, int rows, int k, int p,
                                       const SplitModuli& mods, int8_t* res8, int32_t* shifts, uint32_t* flags,
                                       cudaStream_t stream) {
  return launch_split_mode<true>(X, ldx, rows, k, p, mods, reinterpret_cast<uint8_t*>(res8), shifts, flags, stream);
}

cudaError_t launch_split_rows_s8(const int8_t* X, long long ldx, int rows, int k, uint8_t* planes,
                                 cudaStream_t stream) {
  const int rows_p = round_up(rows, kRowAlign), k_p = round_up(k, kKAlign);
  split_rows_s8_kernel<<<split_grid(rows_p), kSplitThreads, 0, stream>>>(X, ldx, rows, k, rows_p, k_p, planes);
  return cudaGetLastError();
}

cudaError_t launch_transpose_f64(const double* in, long long ldin, int rows, int cols, double* out,
                                 long long ldout, cudaStream_t stream) {
  dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  transpose_kernel<double><<<grid, block, 0, stream>>>(in, ldin, rows, cols, out, ldout);
  return cudaGetLastError();
}

cudaError_t launch_transpose_s8(const int8_t* in, long long ldin, int rows, int cols, int8_t* out, long long ldout,
                                cudaStream_t stream) {
  dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  transpose_kernel<int8_t><<<grid, block, 0, stream>>>(in, ldin, rows, cols, out, ldout);
  return cudaGetLastError();
}

}  // namespace ozemu
