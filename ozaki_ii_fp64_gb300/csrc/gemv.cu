// Fused deconstruction + product for narrow B (n <= 2 columns): the rows of A
// are scaled, rounded and reduced modulo every m_l in registers and dotted
// with B's residues on the spot, so no limb planes of A are written or read.
//
// [TME4] abstract: below the critical intensity OI* the streamed operand's
// deconstruction (the fourth term, c_q r integer instructions per element)
// bounds the emulation; this kernel makes that term as small as it can be:
// per element one scaled integer u = A' + 2^(p_A+1) in two or three 21-bit
// chunks, and per modulus one multiply-add forming t = u (mod m_l) up to a
// multiple of m_l (t < 2^31) plus one 32 x 32 -> 64-bit multiply-add into the
// row's exact sum of t b.  The modular reduction happens once per output:
// sum_k u_k b_k = sum_k A'_k B'_k + 2^(p_A+1) sum_k b_k  (mod m_l).
// The residues c_l written here are those of the FP4 limb path, bit for bit,
// and go through the same CRT kernel.
#include <cstdint>

#include "common.cuh"
#include "deconstruct.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kNarrowThreads = 256;
constexpr int kNarrowColThreads = 512;

// Column j of B (k x n row-major): shift t_j and residues b_{l,k} = B'_kj
// mod m_l in [0, m_l) as bytes at bres[(j R + l) kp + k] (zero for k in
// [k, kp)).
template <int R>
__global__ void __launch_bounds__(kNarrowColThreads) narrow_cols_kernel(const double* __restrict__ B, long long ldb,
                                                                        int k, int kp, int p, const NarrowModuli nm,
                                                                        uint8_t* __restrict__ bres,
                                                                        int32_t* __restrict__ shifts,
                                                                        uint32_t* flags) {
  __shared__ uint64_t red[kNarrowColThreads / 32];
  const int j = blockIdx.x;
  const double* col = B + j;
  uint64_t mx = 0;
  for (int kk = threadIdx.x; kk < k; kk += kNarrowColThreads) {
    const uint64_t a = static_cast<uint64_t>(__double_as_longlong(col[static_cast<long long>(kk) * ldb])) &
                       0x7FFFFFFFFFFFFFFFull;
    mx = a > mx ? a : mx;
  }
  mx = block_max_u64<kNarrowColThreads>(mx, red);
  const int s = mx ? p - frexp_exp_bits(mx) : 0;
  if (mx >= 0x7FF0000000000000ull && threadIdx.x == 0) atomicOr(flags, kFlagNonFinite);
  if (threadIdx.x == 0) shifts[j] = s;

  for (int kk = threadIdx.x; kk < kp; kk += kNarrowColThreads) {
    const uint64_t bits =
        kk < k ? static_cast<uint64_t>(__double_as_longlong(col[static_cast<long long>(kk) * ldb])) : 0ull;
    const uint64_t u = scaled_offset(bits, s);  // B' + 2^62
    const uint32_t a0 = static_cast<uint32_t>(u) & 0x1FFFFFu;
    const uint32_t a1 = static_cast<uint32_t>(u >> 21) & 0x1FFFFFu;
    const uint32_t a2 = static_cast<uint32_t>(u >> 42);
#pragma unroll
    for (int l = 0; l < R; ++l) {
      const uint32_t ml = nm.m[l];
      const uint32_t v = a2 * nm.c42[l] + a1 * nm.c21[l] + a0 + (ml - nm.off62[l]);  // == B' (mod m), < 2^31
      const uint32_t b = v % ml;
      bres[static_cast<long long>(j * R + l) * kp + kk] = static_cast<uint8_t>(b);
    }
  }
}

// |x 2^s| rounded half to even, for the fp64 pattern `bits` of an element of
// a row whose largest magnitude is a normal number, with p <= 52: the scaled
// value is then a right shift of the 53-bit significand by
// d = (1075 - s) - max(E, 1) >= 1.  Non-finite elements give an unspecified
// value (they set the non-finite flag elsewhere).  sgn = -1 or 1.
__device__ __forceinline__ uint64_t rne_right_shift(uint64_t bits, int d0, int& sgn) {
  const uint32_t hi = static_cast<uint32_t>(bits >> 32), lo = static_cast<uint32_t>(bits);
  const uint32_t E = (hi >> 20) & 0x7FFu;
  const uint32_t mhi = (hi & 0xFFFFFu) | (E ? 0x100000u : 0u);
  int d = d0 - static_cast<int>(E > 1u ? E : 1u);
  d = d < 1 ? 1 : (d > 63 ? 63 : d);
  const uint64_t M = (static_cast<uint64_t>(mhi) << 32) | lo;
  const uint64_t q = (M + ((1ull << (d - 1)) - 1ull) + ((M >> d) & 1ull)) >> d;
  sgn = static_cast<int>(hi) >> 31 | 1;
  return q;
}

// One CTA per row of A at a time.  Pass 1 finds the row's exponent, pass 2
// re-reads the row (from L2) and accumulates, for every modulus l and column
// j, S_lj = sum_k t_lk b_{l,k,j} exactly in 64 bits, where t_lk is A'_k in
// signed 21-bit chunks recombined with the weights 2^21, 2^42 mod m_l
// (t == A'_k mod m_l, |t| < 2^30).  Output: c_lj = S_lj mod m_l at
// res[(l m + row) ldr + j] and the row shift.  kTwo: p <= 40, so |A'| <= 2^40
// has two chunks; otherwise p <= 52 and three.
template <int R, int N, bool kTwo, bool kFast>
__device__ __forceinline__ void fused_row_pass(const double* rowp, int k, bool vec_ok, int s, int d0,
                                               const NarrowModuli& nm, const uint8_t* __restrict__ bres, int kp,
                                               long long (&acc)[R][N]) {
  for (int k0 = threadIdx.x * 8; k0 < k; k0 += kNarrowThreads * 8) {
    uint64_t b[8];
    load8_f64(rowp, k, k0, vec_ok, b, true);
    int a0[8], a1[8], a2[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      uint64_t q;
      int sgn;
      if (kFast) {
        q = rne_right_shift(b[e], d0, sgn);
      } else {  // a row whose largest element is subnormal: the general rounding
        const long long v = static_cast<long long>(scaled_offset(b[e], s) - (1ull << 62));
        sgn = v < 0 ? -1 : 1;
        q = static_cast<uint64_t>(v < 0 ? -v : v);
      }
      a0[e] = sgn * static_cast<int>(static_cast<uint32_t>(q) & 0x1FFFFFu);
      if (kTwo) {
        a1[e] = sgn * static_cast<int>(static_cast<uint32_t>(q >> 21));
        a2[e] = 0;
      } else {
        a1[e] = sgn * static_cast<int>(static_cast<uint32_t>(q >> 21) & 0x1FFFFFu);
        a2[e] = sgn * static_cast<int>(static_cast<uint32_t>(q >> 42));
      }
    }
#pragma unroll
    for (int l = 0; l < R; ++l) {
      const int c21 = static_cast<int>(nm.c21[l]), c42 = static_cast<int>(nm.c42[l]);
      uint2 w[N];
#pragma unroll
      for (int j = 0; j < N; ++j)
        w[j] = __ldg(reinterpret_cast<const uint2*>(bres + static_cast<long long>(j * R + l) * kp + k0));
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int t = a1[e] * c21 + a0[e];
        if (!kTwo) t += a2[e] * c42;
#pragma unroll
        for (int j = 0; j < N; ++j) {
          const uint32_t bw = e < 4 ? w[j].x : w[j].y;
          const int bb = static_cast<int>(__byte_perm(bw, 0u, 0x4440u | static_cast<uint32_t>(e & 3)));
          acc[l][j] += static_cast<long long>(t) * bb;
        }
      }
    }
  }
}

template <int R, int N, bool kTwo>
__global__ void __launch_bounds__(kNarrowThreads, N == 1 ? 3 : 2)
    dgemv_fused_kernel(const double* __restrict__ A, long long lda, int m, int k, int kp, int p,
                       const NarrowModuli nm, const uint8_t* __restrict__ bres, uint8_t* __restrict__ res,
                       long long ldr, int32_t* __restrict__ shifts, uint32_t* flags) {
  __shared__ uint64_t red[kNarrowThreads / 32];
  __shared__ long long part[kNarrowThreads / 32][R * N];
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) && ((lda & 1) == 0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int row = blockIdx.x; row < m; row += gridDim.x) {
    const double* rowp = A + static_cast<long long>(row) * lda;
    uint64_t mx = 0;
#pragma unroll 2
    for (int k0 = threadIdx.x * 8; k0 < k; k0 += kNarrowThreads * 8) {
      uint64_t b[8];
      load8_f64(rowp, k, k0, vec_ok, b, false);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint64_t a = b[e] & 0x7FFFFFFFFFFFFFFFull;
        mx = a > mx ? a : mx;
      }
    }
    mx = block_max_u64<kNarrowThreads>(mx, red);
    const int s = mx ? p - frexp_exp_bits(mx) : 0;
    if (mx >= 0x7FF0000000000000ull && threadIdx.x == 0) atomicOr(flags, kFlagNonFinite);

    long long acc[R][N];
#pragma unroll
    for (int l = 0; l < R; ++l)
#pragma unroll
      for (int j = 0; j < N; ++j) acc[l][j] = 0;
    if ((mx >> 52) != 0)  // the row's largest magnitude is normal (or non-finite)
      fused_row_pass<R, N, kTwo, true>(rowp, k, vec_ok, s, 1075 - s, nm, bres, kp, acc);
    else
      fused_row_pass<R, N, kTwo, false>(rowp, k, vec_ok, s, 1075 - s, nm, bres, kp, acc);

#pragma unroll
    for (int l = 0; l < R; ++l)
#pragma unroll
      for (int j = 0; j < N; ++j) {
        long long v = acc[l][j];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0) part[warp][l * N + j] = v;
      }
    __syncthreads();
    if (threadIdx.x < R * N) {
      const int l = threadIdx.x / N, j = threadIdx.x % N;
      long long tot = 0;
#pragma unroll
      for (int w = 0; w < kNarrowThreads / 32; ++w) tot += part[w][threadIdx.x];
      const long long ml = nm.m[l];
      long long c = tot % ml;
      c += c < 0 ? ml : 0;
      res[(static_cast<long long>(l) * m + row) * ldr + j] = static_cast<uint8_t>(c);
    }
    if (threadIdx.x == 0) shifts[row] = s;
  }
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

template <int R>
cudaError_t launch_narrow_r(const NarrowCall& c, cudaStream_t stream) {
  narrow_cols_kernel<R><<<c.n, kNarrowColThreads, 0, stream>>>(c.B, c.ldb, c.k, c.kp, c.pB, c.nm, c.bres, c.sb,
                                                               c.flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int per_sm = c.n == 1 ? 3 : 2;  // the kernels' launch bounds
  const int grid = c.m < sm_count() * per_sm ? c.m : sm_count() * per_sm;
  const bool two = c.pA <= 40;
#define OZEMU_FUSED(NN, TWO)                                                                                     \
  dgemv_fused_kernel<R, NN, TWO><<<grid, kNarrowThreads, 0, stream>>>(c.A, c.lda, c.m, c.k, c.kp, c.pA, c.nm, \
                                                                       c.bres, c.res, c.ldr, c.sa, c.flags)
  if (c.n == 1) {
    if (two)
      OZEMU_FUSED(1, true);
    else
      OZEMU_FUSED(1, false);
  } else {
    if (two)
      OZEMU_FUSED(2, true);
    else
      OZEMU_FUSED(2, false);
  }
#undef OZEMU_FUSED
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_narrow_residues(const NarrowCall& c, cudaStream_t stream) {
  if (c.n < 1 || c.n > kNarrowMaxN || c.k < 1 || c.k > kNarrowMaxK || c.pA > kNarrowMaxP)
    return cudaErrorInvalidValue;
  switch (c.nm.r) {
#define OZEMU_NARROW_CASE(R) \
  case R:                    \
    return launch_narrow_r<R>(c, stream);
    OZEMU_NARROW_CASE(1) OZEMU_NARROW_CASE(2) OZEMU_NARROW_CASE(3) OZEMU_NARROW_CASE(4) OZEMU_NARROW_CASE(5)
    OZEMU_NARROW_CASE(6) OZEMU_NARROW_CASE(7) OZEMU_NARROW_CASE(8) OZEMU_NARROW_CASE(9) OZEMU_NARROW_CASE(10)
    OZEMU_NARROW_CASE(11) OZEMU_NARROW_CASE(12) OZEMU_NARROW_CASE(13) OZEMU_NARROW_CASE(14)
    OZEMU_NARROW_CASE(15) OZEMU_NARROW_CASE(16)
#undef OZEMU_NARROW_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace ozemu
