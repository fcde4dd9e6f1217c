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

constexpr int kNarrowColThreads = 512;

// Column j of B (k x n row-major): shift t_j, residues b_{l,k} = B'_kj mod m_l
// in [0, m_l) as bytes at bres[(j R + l) kp + k] (zero for k in [k, kp)), and
// colsum[j R + l] = sum_k b_{l,k} mod m_l.
template <int R>
__global__ void __launch_bounds__(kNarrowColThreads) narrow_cols_kernel(const double* __restrict__ B, long long ldb,
                                                                        int k, int kp, int p, const NarrowModuli nm,
                                                                        uint8_t* __restrict__ bres,
                                                                        int32_t* __restrict__ colsum,
                                                                        int32_t* __restrict__ shifts,
                                                                        uint32_t* flags) {
  __shared__ uint64_t red[kNarrowColThreads / 32];
  __shared__ uint32_t part[kNarrowColThreads / 32][R];
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

  uint32_t sum[R];
#pragma unroll
  for (int l = 0; l < R; ++l) sum[l] = 0;
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
      sum[l] += b;
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int l = 0; l < R; ++l) {
    uint32_t v = sum[l];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0) part[warp][l] = v;
  }
  __syncthreads();
  if (threadIdx.x < R) {
    uint32_t t = 0;
    for (int w = 0; w < kNarrowColThreads / 32; ++w) t += part[w][threadIdx.x];
    colsum[j * R + threadIdx.x] = static_cast<int32_t>(t % nm.m[threadIdx.x]);
  }
}

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

// Row pass 2 over the thread's elements k0 .. k0 + 7 for k0 in [kbeg, kend),
// for one column of B (bres points at its residues): u_k = A'_k + 2^p in NCH
// unsigned 16-bit chunks, and for every chunk c and modulus l,
// acc[c][l] += sum_k chunk_c(u_k) b_{l,k} with two-way 16 x 8-bit dot
// products (dp2a), four elements per bres word.
template <int R, int NCH, bool kFast, int kThreads>
__device__ __forceinline__ void fused_pass2(const double* rowp, int k, int kbeg, int kend, int vec_ok, int s, int d0,
                                            uint64_t off, const uint8_t* __restrict__ bres, int kp,
                                            uint32_t (&acc)[NCH][R]) {
  for (int k0 = kbeg; k0 < kend; k0 += kThreads * 8) {
    uint64_t b[8];
    load8_f64(rowp, k, k0, vec_ok, b, true);
    uint32_t W[4][NCH];  // element pair q = (2q, 2q + 1): chunk c of both as 16-bit halves
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint64_t u0, u1;
      if (kFast) {
        u0 = offset_integer_fast(b[2 * q], d0, off);
        u1 = offset_integer_fast(b[2 * q + 1], d0, off);
      } else {  // a row whose largest element is subnormal: the general rounding
        u0 = scaled_offset(b[2 * q], s) - (1ull << 62) + off;
        u1 = scaled_offset(b[2 * q + 1], s) - (1ull << 62) + off;
      }
      const uint32_t l0 = static_cast<uint32_t>(u0), l1 = static_cast<uint32_t>(u1);
      const uint32_t h0 = static_cast<uint32_t>(u0 >> 32), h1 = static_cast<uint32_t>(u1 >> 32);
      W[q][0] = __byte_perm(l0, l1, 0x5410);
      W[q][1] = __byte_perm(l0, l1, 0x7632);
      W[q][2] = __byte_perm(h0, h1, 0x5410);
      if (NCH > 3) W[q][3] = __byte_perm(h0, h1, 0x7632);
    }
#pragma unroll
    for (int l = 0; l < R; ++l) {
      const uint2 w = __ldg(reinterpret_cast<const uint2*>(bres + static_cast<long long>(l) * kp + k0));
#pragma unroll
      for (int c = 0; c < NCH; ++c) {
        uint32_t a = acc[c][l];
        a = dp2a_lo(W[0][c], w.x, a);
        a = dp2a_hi(W[1][c], w.x, a);
        a = dp2a_lo(W[2][c], w.y, a);
        a = dp2a_hi(W[3][c], w.y, a);
        acc[c][l] = a;
      }
    }
  }
}

constexpr int kGroup = 256;  // threads that work on one row

__device__ __forceinline__ void group_sync(int bar) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kGroup) : "memory");
}

// Largest value over the group (each thread passes one).
__device__ __forceinline__ uint64_t group_max_u64(uint64_t v, uint64_t* red, int tg, int bar) {
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  group_sync(bar);
  if ((tg & 31) == 0) red[tg >> 5] = v;
  group_sync(bar);
  uint64_t mx = red[0];
#pragma unroll
  for (int w = 1; w < kGroup / 32; ++w) mx = red[w] > mx ? red[w] : mx;
  return mx;
}

// Adds the group's per-thread accumulators (each below 2^30) into tot[]
// (u64, shared memory): sums over lane quads by shuffles (below 2^32), one
// word per quad into buf[64][V + 1], then column sums.
template <int V>
__device__ __forceinline__ void group_sum_into(uint32_t (&v)[V], uint32_t* buf, unsigned long long (*part)[64],
                                               unsigned long long* tot, int tg, int bar) {
  constexpr int kQuads = kGroup / 4;   // 64
  constexpr int kParts = kGroup / 64;  // 4
  constexpr int kStride = V + 1;
  static_assert(V <= 64, "column sums take 64 columns");
#pragma unroll
  for (int i = 0; i < V; ++i) {
    v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], 1);
    v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], 2);
  }
  if ((tg & 3) == 0) {
    uint32_t* row = buf + (tg >> 2) * kStride;
#pragma unroll
    for (int i = 0; i < V; ++i) row[i] = v[i];
  }
  group_sync(bar);
  const int col = tg & 63, prt = tg >> 6;
  if (col < V) {
    unsigned long long sum = 0;
#pragma unroll
    for (int q = 0; q < kQuads / kParts; ++q) sum += buf[(prt * (kQuads / kParts) + q) * kStride + col];
    part[prt][col] = sum;
  }
  group_sync(bar);
  if (tg < V) tot[tg] += part[0][tg] + part[1][tg] + part[2][tg] + part[3][tg];
  group_sync(bar);
}

// One CTA of 256 threads per row at a time, three CTAs per SM: pass 1 finds
// the row's exponent while the other CTAs compute, pass 2 re-reads the row
// from L2 and B's residues through L1 (every row re-reads them, so the
// kernel asks for little shared memory).  The rows in flight (456 x 128 KB
// at K = 16384) fit in L2; prefetching each CTA's next row as well doubled
// that, and pass 2 then missed L2 (0.99 ms against 0.95 ms without).
// Dynamic shared memory: the reduction buffer.
template <int R, int N, int NCH>
__global__ void __launch_bounds__(kGroup, 3)
    dgemv_fused_kernel(const double* __restrict__ A, long long lda, int m, int k, int kp, int p,
                       const NarrowModuli nm, const uint8_t* __restrict__ bres, const int32_t* __restrict__ colsum,
                       uint8_t* __restrict__ res, long long ldr, int32_t* __restrict__ shifts, uint32_t* flags) {
  constexpr int V = N * NCH * R;
  constexpr int kFlushSpan = kGroup * 8 * 8;  // 8 iterations of 8 elements per thread
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ uint64_t red[kGroup / 32];
  __shared__ unsigned long long part[4][64];
  __shared__ unsigned long long tot[V];
  const int tg = threadIdx.x, bar = 1;
  uint32_t* buf = reinterpret_cast<uint32_t*>(dsm);
  const int vec_ok = row_vector_width(A, lda);
  const uint64_t off = 1ull << p;
  const int row_step = gridDim.x;

  for (int row = blockIdx.x; row < m; row += row_step) {
    const double* rowp = A + static_cast<long long>(row) * lda;
    uint64_t mx = 0;
#pragma unroll 4
    for (int k0 = tg * 8; k0 < k; k0 += kGroup * 8) {
      uint64_t b[8];
      load8_f64(rowp, k, k0, vec_ok, b, false);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint64_t a = b[e] & 0x7FFFFFFFFFFFFFFFull;
        mx = a > mx ? a : mx;
      }
    }
    mx = group_max_u64(mx, red, tg, bar);
    const int s = mx ? p - frexp_exp_bits(mx) : 0;
    if (mx >= 0x7FF0000000000000ull && tg == 0) atomicOr(flags, kFlagNonFinite);
    for (int i = tg; i < V; i += kGroup) tot[i] = 0ull;
    const bool fast = (mx >> 52) != 0;  // the row's largest magnitude is normal (or non-finite)
    // Columns one after the other (the second re-reads the row from L2).
    for (int j = 0; j < N; ++j)
      for (int span = 0; span < k; span += kFlushSpan) {
        uint32_t acc[NCH][R];
#pragma unroll
        for (int c = 0; c < NCH; ++c)
#pragma unroll
          for (int l = 0; l < R; ++l) acc[c][l] = 0u;
        const int kbeg = span + tg * 8;
        const int kend = span + kFlushSpan < k ? span + kFlushSpan : k;
        const uint8_t* bj = bres + static_cast<long long>(j) * R * kp;
        if (fast)
          fused_pass2<R, NCH, true, kGroup>(rowp, k, kbeg, kend, vec_ok, s, 1075 - s, off, bj, kp, acc);
        else
          fused_pass2<R, NCH, false, kGroup>(rowp, k, kbeg, kend, vec_ok, s, 1075 - s, off, bj, kp, acc);
        group_sum_into<NCH * R>(reinterpret_cast<uint32_t(&)[NCH * R]>(acc), buf, part, tot + j * NCH * R, tg, bar);
      }

    if (tg < N * R) {
      const int j = tg / R, l = tg % R;
      const unsigned long long ml = nm.m[l];
      unsigned long long c = 0;
#pragma unroll
      for (int ch = 0; ch < NCH; ++ch) c += (tot[(j * NCH + ch) * R + l] % ml) * nm.w16[l][ch];
      c += ml * ml - (static_cast<unsigned long long>(nm.offA[l]) * static_cast<uint32_t>(colsum[j * R + l])) % ml;
      res[(static_cast<long long>(l) * m + row) * ldr + j] = static_cast<uint8_t>(c % ml);
    }
    if (tg == 0) shifts[row] = s;
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
  narrow_cols_kernel<R><<<c.n, kNarrowColThreads, 0, stream>>>(c.B, c.ldb, c.k, c.kp, c.pB, c.nm, c.bres, c.colsum,
                                                               c.sb, c.flags);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const bool three = c.pA <= 46;  // u = A' + 2^p <= 2^47 fits three 16-bit chunks
  const int grid = c.m < sm_count() * 3 ? c.m : sm_count() * 3;  // three CTAs per SM
#define OZEMU_FUSED(NN, NCH)                                                                                      \
  do {                                                                                                          \
    const int dyn = (kGroup / 4) * (NCH * R + 1) * 4;                                                           \
    cudaError_t err = cudaFuncSetAttribute(dgemv_fused_kernel<R, NN, NCH>,                                      \
                                           cudaFuncAttributePreferredSharedMemoryCarveout, 25);                 \
    if (err != cudaSuccess) return err;                                                                         \
    dgemv_fused_kernel<R, NN, NCH><<<grid, kGroup, dyn, stream>>>(c.A, c.lda, c.m, c.k, c.kp, c.pA, c.nm,       \
                                                                  c.bres, c.colsum, c.res, c.ldr, c.sa, c.flags); \
  } while (0)
  if (c.n == 1) {
    if (three)
      OZEMU_FUSED(1, 3);
    else
      OZEMU_FUSED(1, 4);
  } else {
    if (three)
      OZEMU_FUSED(2, 3);
    else
      OZEMU_FUSED(2, 4);
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
