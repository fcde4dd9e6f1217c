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
#include <utility>

#include "common.cuh"
#include "deconstruct.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kSplitThreads = 512;
constexpr int kElemsPerThread = 8;
constexpr int kChunk = kSplitThreads * kElemsPerThread;  // elements of a row per pass step
// Code table: 256 rows (b + 128 for a balanced residue b) of 32 copies of the
// code, word i of a row in bank i.
constexpr int kTableRowShift = 7;
constexpr int kTableRowBytes = 1 << kTableRowShift;
constexpr int kTableWords = 256 * kTableRowBytes / 4;
constexpr int kSplitBlocksPerSM = 2;  // 64 registers x 512 threads; 33 KiB of shared memory each
constexpr int kPrefetchMaxK = 16384;  // longest row whose successor is prefetched into L2

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
  // The nibbles of a pair never overlap: c + (c' << 4) is their bitwise or.
  const uint32_t p01 = c[0] + (c[1] << 4), p23 = c[2] + (c[3] << 4);
  const uint32_t p45 = c[4] + (c[5] << 4), p67 = c[6] + (c[7] << 4);
  uint32_t lo = __byte_perm(p01, p23, 0x5140);
  uint32_t hi = __byte_perm(p45, p67, 0x5140);
  w0 = __byte_perm(lo, hi, 0x5410);
  w1 = __byte_perm(lo, hi, 0x7632);
  uint32_t ulo = __byte_perm(p01, p23, 0x0062);
  uint32_t uhi = __byte_perm(p45, p67, 0x0062);
  w2 = __byte_perm(ulo, uhi, 0x5410);
}

// ---------------------------------------------------------------- residues
// An element's integer A' goes in as u = A' + 2^63 (0 <= u < 2^64), taken as
// its eight bytes: u = sum_i byte_i 2^(8i).  For modulus m, two 4-way byte dot
// products with the weights 2^(8i) mod m (each < 256) and an accumulator
// bias give v = u + bias < 2^20 with v = A' + h (mod m), h = floor(m/2).  The
// quotient floor(v/m) comes from one fp32 fma rounded down: v and 2^23 are
// exact in fp32, 1/m is taken rounded up (c = ceil(2^e/m) 2^-e with
// e = 23 + ceil(log2 m), a 24-bit integer times a power of two), and
// v c - v/m < 2^(20-e) <= 2^-9 < 1/m, so rd(v c + 2^23) = 2^23 + floor(v/m)
// exactly; its bit pattern is 0x4B000000 + floor(v/m).  (An even modulus
// other than 256, 112 in the two-limb list, takes an exact Barrett step with
// ceil(2^32/m) instead, v m < 2^32.)  Then w = v - m floor(v/m) is
// (A' + h) mod m and b = w - h is the balanced residue, in [-h, m - 1 - h] as
// the method takes it.  The codes of b come from one table shared by every
// modulus, indexed by b + 128.
__host__ __device__ constexpr uint32_t pow2_mod(int e, uint32_t m) {
  uint64_t r = 1 % m;
  for (int i = 0; i < e; ++i) r = r * 2 % m;
  return static_cast<uint32_t>(r);
}

struct ResidueStep {
  uint32_t m, clo, chi, bias, row;
  float inv_up;
};

// Modulus l of the 3-limb (nl = 3), two-limb (nl = 2) or mixed-digit
// (nl = 1) list.
__host__ __device__ constexpr uint32_t table_modulus(int l, int nl) {
  return nl == 1 ? kModulusTableMix[l] : (nl == 2 ? kModulusTable2[l] : kModulusTable[l]);
}

// Table rows 0 .. 10 (residues b < -117, which no modulus of the mixed-digit
// list reaches) hold, in the mixed-digit launch, the single digit of each
// residue modulo 11: row w for b = w - 5, the member of S congruent to b
// mod 11 of smallest magnitude (b = +-5 -> -+6).  Every other single-digit
// modulus takes the low base-13 digit of the shared rows, which is b itself
// for |b| <= 4 and the class digit mod 13 (b = +-5, +-6 -> -+8, 6, -6) for 13.
constexpr uint32_t kMod11Row = 0u;

__host__ __device__ constexpr ResidueStep residue_step(int l, int nl) {
  const uint32_t m = table_modulus(l, nl), h = m >> 1;
  ResidueStep st{m, 0u, 0u, 0u, 0u, 0.0f};
  for (int i = 0; i < 4; ++i) {
    st.clo |= pow2_mod(8 * i, m) << (8 * i);
    st.chi |= pow2_mod(32 + 8 * i, m) << (8 * i);
  }
  st.bias = (h + m - pow2_mod(63, m)) % m;
  st.row = (nl == 1 && m == 11u) ? kMod11Row : 128u - h;  // table row of b = -h
  int lg = 0;
  while ((1u << lg) < m) ++lg;
  const int e = 23 + lg;  // ceil(2^e / m) lies in [2^23, 2^24): exact in fp32
  st.inv_up = static_cast<float>(((1ull << e) + m - 1) / m) / static_cast<float>(1ull << e);
  return st;
}

// The per-modulus constants in the constant bank (operands of the dot
// products and the fma), with the dot-product bias carrying 0x4B000000 for
// the odd moduli (the fp32 quotient).
__host__ __device__ constexpr ResidueStep residue_step_biased(int l, int nl) {
  ResidueStep st = residue_step(l, nl);
  if (st.m % 2 == 1) st.bias += 0x4B000000u;
  return st;
}
#define OZEMU_STEPS(NL)                                                                                      \
  {residue_step_biased(0, NL),  residue_step_biased(1, NL),  residue_step_biased(2, NL),                    \
   residue_step_biased(3, NL),  residue_step_biased(4, NL),  residue_step_biased(5, NL),                    \
   residue_step_biased(6, NL),  residue_step_biased(7, NL),  residue_step_biased(8, NL),                    \
   residue_step_biased(9, NL),  residue_step_biased(10, NL), residue_step_biased(11, NL),                   \
   residue_step_biased(12, NL), residue_step_biased(13, NL), residue_step_biased(14, NL),                   \
   residue_step_biased(15, NL)}
__constant__ ResidueStep kSteps3[kMaxModuli] = OZEMU_STEPS(3);
__constant__ ResidueStep kSteps2[kMaxModuli] = OZEMU_STEPS(2);
__constant__ ResidueStep kSteps1[kMaxModuliMix] = {
    residue_step_biased(0, 1),  residue_step_biased(1, 1),  residue_step_biased(2, 1),  residue_step_biased(3, 1),
    residue_step_biased(4, 1),  residue_step_biased(5, 1),  residue_step_biased(6, 1),  residue_step_biased(7, 1),
    residue_step_biased(8, 1),  residue_step_biased(9, 1),  residue_step_biased(10, 1), residue_step_biased(11, 1),
    residue_step_biased(12, 1), residue_step_biased(13, 1), residue_step_biased(14, 1), residue_step_biased(15, 1),
    residue_step_biased(16, 1), residue_step_biased(17, 1), residue_step_biased(18, 1), residue_step_biased(19, 1)};
#undef OZEMU_STEPS

// Digits per modulus: NL for the 3- and two-limb lists; in the mixed-digit
// list (NL = 1) one for the first kMixSingle moduli and two for the rest.
template <int L, int NL>
__host__ __device__ constexpr int digits_of() {
  return NL == 1 ? (L < kMixSingle ? 1 : 2) : NL;
}

// Byte offset of this lane's table word for the balanced residue of A'
// modulo modulus L, relative to the table row of b = -h.  A table row is 128
// bytes: lane i's copy of the code at bytes 4i (bank i).  lane_hi =
// (4 lane) << 25: the funnel shift puts w at bit 7 and the lane's word at bits
// 2..6.  With the fp32 quotient,
// vb - m (0x4B000000 + floor(v/m)) = w + 0x4B000000 (1 - m) (mod 2^32), and
// for odd m, 0x4B000000 (1 - m) 2^7 = 0 (mod 2^32), so the shifted value is
// w's (m = 256 takes the low byte directly).
template <int L, int NL>
__device__ __forceinline__ uint32_t residue_offset(uint32_t ulo, uint32_t uhi, uint32_t lane_hi) {
  constexpr ResidueStep st = residue_step(L, NL);
  const ResidueStep& ks = NL == 1 ? kSteps1[L] : (NL == 2 ? kSteps2[L] : kSteps3[L]);
  uint32_t w;
  if constexpr (st.m == 256u) {
    w = (ulo & 0xFFu) ^ 0x80u;  // 2^63 = 0 (mod 256): b is the low byte of A', signed
  } else if constexpr (st.m % 2 == 0) {
    const uint32_t v = __dp4a(ulo, ks.clo, __dp4a(uhi, ks.chi, ks.bias));
    constexpr uint32_t kMagic = static_cast<uint32_t>(((1ull << 32) + st.m - 1) / st.m);
    w = v - __umulhi(v, kMagic) * st.m;
  } else {
    // vb = 0x4B000000 + v: the fp32 pattern of 2^23 + v (v < 2^23).
    const uint32_t vb = __dp4a(ulo, ks.clo, __dp4a(uhi, ks.chi, ks.bias));
    const float vf = __uint_as_float(vb) - 8388608.0f;
    const uint32_t qb = __float_as_uint(__fmaf_rd(vf, ks.inv_up, 8388608.0f));
    w = vb - qb * st.m;
  }
  return __funnelshift_l(lane_hi, w, kTableRowShift);
}

// Codes of 8 elements for modulus L, packed and stored.  Lane i reads bank i
// only, so a warp's lookups never conflict.  o / modulus_words: this row's
// word of modulus 0 and the stride between moduli; in the mixed-digit list
// the single-digit moduli use (o, modulus_words) and the two-digit ones
// (o2, modulus_words2), counted from the first two-digit modulus.
template <int L, bool kRes8, int NL>
__device__ __forceinline__ void modulus_codes(const uint32_t (&ulo)[8], const uint32_t (&uhi)[8], const char* tb,
                                              uint32_t lane_hi, uint32_t* o, long long modulus_words, uint32_t* o2,
                                              long long modulus_words2) {
  constexpr uint32_t kRow0 = residue_step(L, NL).row * kTableRowBytes;
  const char* t0 = tb + kRow0;
  uint32_t c[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    c[e] = *reinterpret_cast<const uint32_t*>(t0 + residue_offset<L, NL>(ulo[e], uhi[e], lane_hi));
  }
  if constexpr (kRes8) {
    uint2 w;
    w.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    w.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
    __stcs(reinterpret_cast<uint2*>(o + L * modulus_words), w);
  } else {
    uint32_t w0, w1, w2;
    pack8(c, w0, w1, w2);
    // Limb j of a 128-element K block sits 64 j bytes after limb 0 (two-limb
    // moduli: the third limb is 0 and not stored; single-digit moduli store
    // the low digit only).
    constexpr int D = digits_of<L, NL>();
    uint32_t* p = (NL == 1 && L >= kMixSingle) ? o2 + (L - kMixSingle) * modulus_words2 : o + L * modulus_words;
    __stcs(p, w0);
    if constexpr (D >= 2) __stcs(p + 16, w1);
    if constexpr (D == 3) __stcs(p + 32, w2);
  }
}

template <bool kRes8, int NL, int... Ls>
__device__ __forceinline__ void all_moduli(std::integer_sequence<int, Ls...>, const uint32_t (&ulo)[8],
                                           const uint32_t (&uhi)[8], const char* tb, uint32_t lane_hi, uint32_t* o,
                                           long long modulus_words, uint32_t* o2, long long modulus_words2) {
  (modulus_codes<Ls, kRes8, NL>(ulo, uhi, tb, lane_hi, o, modulus_words, o2, modulus_words2), ...);
}

// Pass 2 of the row split over the row's elements: integers, residues and
// limb codes (or residue bytes), packed and stored.  out_row2 /
// modulus_words2: the row of the first two-digit modulus and the stride
// between two-digit moduli (mixed-digit list only).
template <int R, bool kRes8, int NL, bool kFast>
__device__ __forceinline__ void split_pass2(const double* rowp, int k, int k_p, int vec_ok, int s, const char* tb,
                                            uint32_t lane_hi, uint8_t* out_row, long long modulus_words,
                                            uint8_t* out_row2, long long modulus_words2) {
  // Backwards over the row: pass 1 read it forwards, so the most recently
  // read part (the likeliest still in L2) comes first.
  const int kfirst = threadIdx.x * kElemsPerThread;
  const int klast = kfirst < k_p ? kfirst + ((k_p - 1 - kfirst) / kChunk) * kChunk : -1;
  for (int k0 = klast; k0 >= kfirst; k0 -= kChunk) {
    uint64_t b[8];
    load8_f64(rowp, k, k0, vec_ok, b, true);
    uint32_t ulo[8], uhi[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint64_t u =
          kFast ? offset_integer_fast(b[e], 1075 - s, 1ull << 63) : scaled_offset(b[e], s) + (1ull << 62);
      ulo[e] = static_cast<uint32_t>(u);
      uhi[e] = static_cast<uint32_t>(u >> 32);
    }
    // Single-digit rows (mixed list) hold one 64-byte digit run per K block.
    constexpr int kRun = NL == 1 ? 64 : 64 * NL;
    uint32_t* o = reinterpret_cast<uint32_t*>(out_row + (kRes8 ? k0 : (k0 >> 7) * kRun + (k0 & 127) / 2));
    uint32_t* o2 = NL == 1 ? reinterpret_cast<uint32_t*>(out_row2 + (k0 >> 7) * 128 + (k0 & 127) / 2) : nullptr;
    all_moduli<kRes8, NL>(std::make_integer_sequence<int, R>{}, ulo, uhi, tb, lane_hi, o, modulus_words, o2,
                          modulus_words2);
  }
}

// Largest (high word & 0x7FFFFFFF) over a row: the high word of the largest
// magnitude.  With 32-byte rows each load instruction of a warp covers 1 KiB
// of consecutive addresses, four of them in flight per thread.
__device__ __forceinline__ uint32_t row_max_hi(const double* rowp, int k, int vec) {
  uint32_t mh = 0;
  if (vec == 2) {
    constexpr int kStep = kSplitThreads * 4;
    int k0 = threadIdx.x * 4;
    for (; k0 + 3 * kStep + 4 <= k; k0 += 4 * kStep) {
      uint32_t h[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        unsigned long long x0, x1, x2, x3;
        asm volatile("ld.global.nc.v4.u64 {%0, %1, %2, %3}, [%4];"
                     : "=l"(x0), "=l"(x1), "=l"(x2), "=l"(x3)
                     : "l"(rowp + k0 + q * kStep));
        h[4 * q] = static_cast<uint32_t>(x0 >> 32);
        h[4 * q + 1] = static_cast<uint32_t>(x1 >> 32);
        h[4 * q + 2] = static_cast<uint32_t>(x2 >> 32);
        h[4 * q + 3] = static_cast<uint32_t>(x3 >> 32);
      }
#pragma unroll
      for (int i = 0; i < 16; i += 2) mh = __vimax3_u32(mh, h[i] & 0x7FFFFFFFu, h[i + 1] & 0x7FFFFFFFu);
    }
    for (; k0 + 4 <= k; k0 += kStep) {
      unsigned long long x0, x1, x2, x3;
      asm volatile("ld.global.nc.v4.u64 {%0, %1, %2, %3}, [%4];"
                   : "=l"(x0), "=l"(x1), "=l"(x2), "=l"(x3)
                   : "l"(rowp + k0));
      mh = __vimax3_u32(mh, static_cast<uint32_t>(x0 >> 32) & 0x7FFFFFFFu, static_cast<uint32_t>(x1 >> 32) & 0x7FFFFFFFu);
      mh = __vimax3_u32(mh, static_cast<uint32_t>(x2 >> 32) & 0x7FFFFFFFu, static_cast<uint32_t>(x3 >> 32) & 0x7FFFFFFFu);
    }
    for (; k0 < k; ++k0) mh = max(mh, static_cast<uint32_t>(__double_as_longlong(rowp[k0]) >> 32) & 0x7FFFFFFFu);
  } else {
    for (int i = threadIdx.x; i < k; i += kSplitThreads)
      mh = max(mh, static_cast<uint32_t>(__double_as_longlong(rowp[i]) >> 32) & 0x7FFFFFFFu);
  }
  return mh;
}

template <int kThreads>
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t m = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) m = max(m, red[w]);
  return m;
}

// Single digit of a balanced residue b modulo 11 (|b| <= 5): b itself, or
// -+6 for b = +-5 (the members of S congruent to b mod 11).
__device__ uint32_t mod11_code(int b) {
  const int d = b == 5 ? -6 : (b == -5 ? 6 : b);
  return e2m1_nibble(d);
}

// kRes8 = false: FP4 limb planes [r][3][rows_p][k_p/2] (the FP4 path).
// kRes8 = true: the balanced residues themselves as int8 [r][rows_p][k_p]
// (input of the INT8 comparison GEMM).  NL = 1: the mixed-digit list, whose
// single-digit moduli come first ([l][rows_p][k_p/2] each) and whose
// two-digit moduli follow ([l][rows_p][k_p] each, the two-limb layout).
template <int R, bool kRes8, int NL>
__global__ void __launch_bounds__(kSplitThreads, kSplitBlocksPerSM)
    split_rows_f64_kernel(const double* __restrict__ X, long long ldx, int rows, int k, int rows_p, int k_p, int p,
                          uint8_t* __restrict__ planes, int32_t* __restrict__ shifts, uint32_t* flags) {
  // Code table: row j = 32 copies of the codes (or residue byte) of
  // b = j - 128, word i read by lane i; then 256 words of staging.
  extern __shared__ __align__(16) uint32_t tbl[];
  __shared__ uint32_t red[kSplitThreads / 32];
  uint32_t* stage = tbl + kTableWords;
  for (int i = threadIdx.x; i < 256; i += kSplitThreads) {
    uint32_t code = kRes8 ? static_cast<uint32_t>(static_cast<uint8_t>(i - 128)) : limb_code(i - 128);
    if (NL == 1 && i >= static_cast<int>(kMod11Row) && i < static_cast<int>(kMod11Row) + 11)
      code = mod11_code(i - static_cast<int>(kMod11Row) - 5);
    stage[i] = code;
  }
  __syncthreads();
  for (int w = threadIdx.x; w < kTableWords; w += kSplitThreads)
    tbl[w] = stage[w >> (kTableRowShift - 2)];
  __syncthreads();
  const char* tb = reinterpret_cast<const char*>(tbl);
  const uint32_t lane_hi = (threadIdx.x & 31u) << (34 - kTableRowShift);  // (4 lane) << 25

  // FP4 planes: a row holds the three limbs of each 128-element K block
  // side by side (3 x 64 bytes); moduli follow one another.  Mixed-digit
  // list: single-digit rows of k_p/2 bytes, then two-digit rows of k_p.
  const long long row_bytes = kRes8 ? k_p : static_cast<long long>(NL) * k_p / 2;
  const long long modulus_stride = static_cast<long long>(rows_p) * row_bytes;
  constexpr int kSingle = NL == 1 ? (R < kMixSingle ? R : kMixSingle) : 0;  // mixed: single-digit moduli
  const long long row_bytes2 = k_p;
  const long long modulus_stride2 = static_cast<long long>(rows_p) * row_bytes2;
  uint8_t* planes2 = planes + kSingle * modulus_stride;  // first two-digit modulus (mixed list)
  const int vec_ok = row_vector_width(X, ldx);

  for (int row = blockIdx.x; row < rows_p; row += gridDim.x) {
    uint8_t* out_row = planes + static_cast<long long>(row) * row_bytes;
    uint8_t* out_row2 = planes2 + static_cast<long long>(row) * row_bytes2;
    if (row >= rows) {  // padding row: digit (or residue) 0 everywhere
      for (int l = 0; l < R; ++l) {
        const bool two = NL == 1 && l >= kSingle;
        uint32_t* o = reinterpret_cast<uint32_t*>(two ? out_row2 + (l - kSingle) * modulus_stride2
                                                      : out_row + l * modulus_stride);
        const long long words = (two ? row_bytes2 : row_bytes) / 4;
        for (int w = threadIdx.x; w < words; w += kSplitThreads) o[w] = 0u;
      }
      continue;
    }
    const double* rowp = X + static_cast<long long>(row) * ldx;

    // Pass 1: exponent of the largest magnitude of the row.  The high words
    // decide it unless every high word is zero (magnitudes below 2^-1042),
    // when the low words are scanned too.
    const uint32_t mh = block_max_u32<kSplitThreads>(row_max_hi(rowp, k, vec_ok), red);
    int s = 0;
    if (mh >= 0x00100000u) {
      s = p - (static_cast<int>(mh >> 20) - 1022);
    } else if (mh != 0) {
      s = p - ((64 - __clz(static_cast<int>(mh))) - 1074);
    } else {
      uint32_t ml = 0;
      for (int i = threadIdx.x; i < k; i += kSplitThreads)
        ml = max(ml, static_cast<uint32_t>(__double_as_longlong(rowp[i])));
      ml = block_max_u32<kSplitThreads>(ml, red);
      if (ml != 0) s = p - ((32 - __clz(static_cast<int>(ml))) - 1074);
    }
    if (mh >= 0x7FF00000u && threadIdx.x == 0) atomicOr(flags, kFlagNonFinite);
    if (threadIdx.x == 0) shifts[row] = s;

    // Bring this CTA's next row into L2 while this one is split, when the
    // current and next rows of every resident CTA fit in L2 together
    // (2 x 304 CTAs x 16384 x 8 B = 80 MB); longer rows would evict the
    // current row before pass 2 re-reads it.
    if (k <= kPrefetchMaxK && row + static_cast<int>(gridDim.x) < rows) {
      const double* nrow = rowp + static_cast<long long>(gridDim.x) * ldx;
      for (int k0 = threadIdx.x * 16; k0 < k; k0 += kSplitThreads * 16)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(nrow + k0));
    }

    // Pass 2: integers, residues, limbs.  Rows whose largest magnitude is
    // normal (with p <= 52) take the right-shift rounding.
    if (mh >= 0x00100000u && p <= 52)
      split_pass2<R, kRes8, NL, true>(rowp, k, k_p, vec_ok, s, tb, lane_hi, out_row, modulus_stride / 4, out_row2,
                                      modulus_stride2 / 4);
    else
      split_pass2<R, kRes8, NL, false>(rowp, k, k_p, vec_ok, s, tb, lane_hi, out_row, modulus_stride / 4, out_row2,
                                       modulus_stride2 / 4);
  }
}

__global__ void __launch_bounds__(kSplitThreads) split_rows_s8_kernel(const int8_t* __restrict__ X, long long ldx,
                                                                     int rows, int k, int rows_p, int k_p,
                                                                     uint8_t* __restrict__ planes) {
  __shared__ uint32_t lut[256];
  for (int i = threadIdx.x; i < 256; i += kSplitThreads) lut[i] = limb_code(i - 128);
  __syncthreads();
  const long long row_bytes = 3LL * k_p / 2;  // the three limbs of each 128-element K block side by side
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
      uint32_t* o = o_row + (k0 >> 7) * 48 + (k0 & 127) / 8;
      o[0] = w0;
      o[16] = w1;
      o[32] = w2;
    }
  }
}

// INT8 limb planes of the columns of X (k x cols, row-major): column j
// becomes plane row j, without a transposed copy.  One CTA per (128-element
// K block, 64 columns): the block is staged in shared memory as it lies in
// X (coalesced 4-byte loads along the rows), each thread forms the codes of
// 32 consecutive K elements of one column, and the 4 lanes of a column write
// its 64-byte run of each limb with one 16-byte store each.  Padding columns
// (cols <= j < cols_p) and K elements (k <= e < k_p) get code 0.
constexpr int kColTile = 64;
constexpr int kColPitch = kColTile + 4;  // bytes per staged K row

__global__ void __launch_bounds__(256) split_cols_s8_kernel(const int8_t* __restrict__ X, long long ldx, int k,
                                                            int cols, int k_p, uint8_t* __restrict__ planes) {
  __shared__ uint32_t lut[256];
  __shared__ __align__(16) uint8_t tile[128 * kColPitch];
  lut[threadIdx.x] = limb_code(static_cast<int>(threadIdx.x) - 128);
  const int c0 = blockIdx.x * kColTile;
  const int kb = blockIdx.y;
  const bool vec = ((reinterpret_cast<uintptr_t>(X) & 3u) == 0) && ((ldx & 3) == 0) && (c0 + kColTile <= cols);
  for (int w = threadIdx.x; w < 128 * (kColTile / 4); w += 256) {
    const int i = w / (kColTile / 4), q = w % (kColTile / 4);
    const int kr = kb * 128 + i;
    uint32_t v = 0;
    if (kr < k) {
      const int8_t* src = X + static_cast<long long>(kr) * ldx + c0 + 4 * q;
      if (vec) {
        v = __ldg(reinterpret_cast<const unsigned int*>(src));
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c0 + 4 * q + e < cols) v |= static_cast<uint32_t>(static_cast<uint8_t>(src[e])) << (8 * e);
      }
    }
    *reinterpret_cast<uint32_t*>(tile + i * kColPitch + 4 * q) = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int col = (threadIdx.x >> 5) * 8 + (lane >> 2);  // column within the tile, 0..63
  const int q = lane & 3;                                // K elements 32 q .. 32 q + 31 of the block
  uint32_t w[3][4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      c[e] = lut[static_cast<int>(static_cast<int8_t>(tile[(q * 32 + g * 8 + e) * kColPitch + col])) + 128];
    pack8(c, w[0][g], w[1][g], w[2][g]);
  }
  uint8_t* o = planes + static_cast<long long>(c0 + col) * (3LL * k_p / 2) + kb * 192 + q * 16;
#pragma unroll
  for (int l = 0; l < 3; ++l)
    *reinterpret_cast<uint4*>(o + l * 64) = make_uint4(w[l][0], w[l][1], w[l][2], w[l][3]);
}

// ------------------------------------------------- INT4 x INT8, four planes
// Packs 8 four-plane codes (nibble of plane j in byte j) into the four plane
// words: word j holds plane j of elements 0..7, element e in nibble e.
__device__ __forceinline__ void pack8_four(const uint32_t (&c)[8], uint32_t (&w)[4]) {
  const uint32_t p01 = c[0] + (c[1] << 4), p23 = c[2] + (c[3] << 4);
  const uint32_t p45 = c[4] + (c[5] << 4), p67 = c[6] + (c[7] << 4);
  const uint32_t lo = __byte_perm(p01, p23, 0x5140), hi = __byte_perm(p45, p67, 0x5140);
  const uint32_t lo2 = __byte_perm(p01, p23, 0x7362), hi2 = __byte_perm(p45, p67, 0x7362);
  w[0] = __byte_perm(lo, hi, 0x5410);
  w[1] = __byte_perm(lo, hi, 0x7632);
  w[2] = __byte_perm(lo2, hi2, 0x5410);
  w[3] = __byte_perm(lo2, hi2, 0x7632);
}

// Code of an int8 value from the four-plane table; a value the table marks
// out of range (0xFFFFFFFF) raises kFlagRange and takes digit 0.
__device__ __forceinline__ uint32_t four_code(const uint32_t* lut, int v, bool& bad) {
  const uint32_t c = lut[v + 128];
  bad |= (c == 0xFFFFFFFFu);
  return c == 0xFFFFFFFFu ? 0u : c;
}

// Four planes of the rows of X (rows x k, int8, row-major): row i of the
// planes holds, per 128-element K block, the 64 bytes of each of the four
// planes side by side; padding rows and K elements get code 0.
__global__ void __launch_bounds__(kSplitThreads) split_rows_four_kernel(const int8_t* __restrict__ X, long long ldx,
                                                                       int rows, int k, int rows_p, int k_p,
                                                                       uint8_t* __restrict__ planes,
                                                                       const __grid_constant__ FourCodes codes,
                                                                       uint32_t* flags) {
  __shared__ uint32_t lut[256];
  for (int i = threadIdx.x; i < 256; i += kSplitThreads) lut[i] = codes.code[i];
  __syncthreads();
  const long long row_bytes = 2LL * k_p;
  const bool vec_ok = ((reinterpret_cast<uintptr_t>(X) & 7u) == 0) && ((ldx & 7) == 0);
  bool bad = false;
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
      uint32_t c[8], w[4];
#pragma unroll
      for (int e = 0; e < 8; ++e) c[e] = four_code(lut, v[e], bad);
      pack8_four(c, w);
      uint32_t* o = o_row + (k0 >> 7) * 64 + (k0 & 127) / 8;
#pragma unroll
      for (int j = 0; j < 4; ++j) o[16 * j] = w[j];
    }
  }
  if (bad) atomicOr(flags, kFlagRange);
}

// Four planes of the columns of X (k x cols, int8, row-major): plane row j
// holds column j.  One CTA per (128-element K block, 64 columns), staged in
// shared memory as in split_cols_s8_kernel.
__global__ void __launch_bounds__(256) split_cols_four_kernel(const int8_t* __restrict__ X, long long ldx, int k,
                                                              int cols, int k_p, uint8_t* __restrict__ planes,
                                                              const __grid_constant__ FourCodes codes,
                                                              uint32_t* flags) {
  __shared__ uint32_t lut[256];
  __shared__ __align__(16) uint8_t tile[128 * (64 + 4)];
  constexpr int kPitch = 64 + 4;
  lut[threadIdx.x] = codes.code[threadIdx.x];
  const int c0 = blockIdx.x * 64;
  const int kb = blockIdx.y;
  const bool vec = ((reinterpret_cast<uintptr_t>(X) & 3u) == 0) && ((ldx & 3) == 0) && (c0 + 64 <= cols);
  for (int w = threadIdx.x; w < 128 * 16; w += 256) {
    const int i = w / 16, q = w % 16;
    const int kr = kb * 128 + i;
    uint32_t v = 0;
    if (kr < k) {
      const int8_t* src = X + static_cast<long long>(kr) * ldx + c0 + 4 * q;
      if (vec) {
        v = __ldg(reinterpret_cast<const unsigned int*>(src));
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c0 + 4 * q + e < cols) v |= static_cast<uint32_t>(static_cast<uint8_t>(src[e])) << (8 * e);
      }
    }
    *reinterpret_cast<uint32_t*>(tile + i * kPitch + 4 * q) = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int col = (threadIdx.x >> 5) * 8 + (lane >> 2);  // column within the tile, 0..63
  const int q = lane & 3;                                // K elements 32 q .. 32 q + 31 of the block
  bool bad = false;
  uint32_t w[4][4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    uint32_t c[8], wg[4];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      c[e] = four_code(lut, static_cast<int>(static_cast<int8_t>(tile[(q * 32 + g * 8 + e) * kPitch + col])), bad);
    pack8_four(c, wg);
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j][g] = wg[j];
  }
  uint8_t* o = planes + static_cast<long long>(c0 + col) * (2LL * k_p) + kb * 256 + q * 16;
#pragma unroll
  for (int j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(o + j * 64) = make_uint4(w[j][0], w[j][1], w[j][2], w[j][3]);
  if (bad) atomicOr(flags, kFlagRange);
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

// ------------------------------------------------------------- fp64 columns
// Columns of X (k x cols, row-major) split without a transposed copy, in two
// passes over X: the column maxima, then persistent CTAs that each take
// (64 columns, 128-row K block) items: the block is staged in shared memory
// column by column (each warp loads 32 consecutive elements of a row), and
// 16 threads of a column form the digit words of its 16 runs of 8 K elements,
// so a warp's stores are two 64-byte runs of plane rows, as the row split's
// stores are 128-byte runs.
constexpr int kColStrip = 64;       // columns per work item
constexpr int kColPitchF64 = 129;   // doubles per staged column (odd: loads/stores at most 2 wavefronts per 256 B)
constexpr int kColMaxRows = 128;    // rows per CTA of the column-maximum pass
constexpr int kColThreads = 512;

// colmax[j] = max over column j of |x| as a 63-bit pattern (atomicMax into a
// zeroed array): warp w of a CTA reads rows r0 + w, r0 + w + 8, ..., each
// lane two adjacent columns of a 64-column strip.
__global__ void __launch_bounds__(256) col_absmax_kernel(const double* __restrict__ X, long long ldx, int k,
                                                         int cols, unsigned long long* __restrict__ colmax) {
  __shared__ unsigned long long part[8][kColStrip];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c0 = blockIdx.x * kColStrip;
  const int r0 = blockIdx.y * kColMaxRows;
  const int r1 = min(r0 + kColMaxRows, k);
  const int col = c0 + 2 * lane;
  const bool vec = ((reinterpret_cast<uintptr_t>(X) & 15u) == 0) && ((ldx & 1) == 0) && (col + 1 < cols);
  unsigned long long m0 = 0, m1 = 0;
  for (int row = r0 + warp; row < r1; row += 8) {
    const double* p = X + static_cast<long long>(row) * ldx + col;
    unsigned long long b0 = 0, b1 = 0;
    if (vec) {
      const double2 v = *reinterpret_cast<const double2*>(p);
      b0 = static_cast<unsigned long long>(__double_as_longlong(v.x));
      b1 = static_cast<unsigned long long>(__double_as_longlong(v.y));
    } else {
      if (col < cols) b0 = static_cast<unsigned long long>(__double_as_longlong(p[0]));
      if (col + 1 < cols) b1 = static_cast<unsigned long long>(__double_as_longlong(p[1]));
    }
    b0 &= 0x7FFFFFFFFFFFFFFFull;
    b1 &= 0x7FFFFFFFFFFFFFFFull;
    m0 = b0 > m0 ? b0 : m0;
    m1 = b1 > m1 ? b1 : m1;
  }
  part[warp][2 * lane] = m0;
  part[warp][2 * lane + 1] = m1;
  __syncthreads();
  if (threadIdx.x < kColStrip && c0 + static_cast<int>(threadIdx.x) < cols) {
    unsigned long long m = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) m = part[w][threadIdx.x] > m ? part[w][threadIdx.x] : m;
    if (m) atomicMax(colmax + c0 + threadIdx.x, m);
  }
}

// The digit words of 8 K elements (staged column pointer src) of one column
// for every modulus: the fast rounding or the general one.
template <int R, int NL, bool kFast>
__device__ __forceinline__ void col_words(const double* src, int rot, int s, const char* tb, uint32_t lane_hi,
                                          uint32_t* o, long long mw, uint32_t* o2, long long mw2) {
  uint32_t ulo[8], uhi[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(src[(e + rot) & 7]));
    const uint64_t u = kFast ? offset_integer_fast(bits, 1075 - s, 1ull << 63) : scaled_offset(bits, s) + (1ull << 62);
    ulo[e] = static_cast<uint32_t>(u);
    uhi[e] = static_cast<uint32_t>(u >> 32);
  }
  all_moduli<false, NL>(std::make_integer_sequence<int, R>{}, ulo, uhi, tb, lane_hi, o, mw, o2, mw2);
}

template <int R, int NL>
__global__ void __launch_bounds__(kColThreads, 2)
    split_cols_f64_kernel(const double* __restrict__ X, long long ldx, int k, int cols, int cols_p, int k_p, int p,
                          const unsigned long long* __restrict__ colmax, uint8_t* __restrict__ planes,
                          int32_t* __restrict__ shifts, uint32_t* flags) {
  extern __shared__ __align__(16) uint32_t tbl[];
  uint32_t* stage = tbl + kTableWords;
  double* tile = reinterpret_cast<double*>(stage + 256);  // [kColStrip][kColPitchF64]: column c at tile + c * pitch
  for (int i = threadIdx.x; i < 256; i += kColThreads) {
    uint32_t code = limb_code(i - 128);
    if (NL == 1 && i >= static_cast<int>(kMod11Row) && i < static_cast<int>(kMod11Row) + 11)
      code = mod11_code(i - static_cast<int>(kMod11Row) - 5);
    stage[i] = code;
  }
  __syncthreads();
  for (int w = threadIdx.x; w < kTableWords; w += kColThreads) tbl[w] = stage[w >> (kTableRowShift - 2)];
  const char* tb = reinterpret_cast<const char*>(tbl);
  const uint32_t lane_hi = (threadIdx.x & 31u) << (34 - kTableRowShift);

  // Plane rows as the row split writes them (single-digit rows of the mixed
  // list first, then its two-digit rows).
  const long long row_bytes = static_cast<long long>(NL) * k_p / 2;
  const long long modulus_stride = static_cast<long long>(cols_p) * row_bytes;
  constexpr int kSingle = NL == 1 ? (R < kMixSingle ? R : kMixSingle) : 0;
  const long long row_bytes2 = k_p;
  const long long modulus_stride2 = static_cast<long long>(cols_p) * row_bytes2;
  constexpr int kRun = NL == 1 ? 64 : 64 * NL;
  const int wd = threadIdx.x & 15;    // word of the 64-byte digit run: K elements 8 wd .. 8 wd + 7
  const int cl = threadIdx.x >> 4;    // column within a 32-column half of the strip
  const int nstrips = cols_p / kColStrip;
  const int total = nstrips * (k_p / 128);

  // Work item w: (64-column strip w % nstrips, K block w / nstrips), so
  // neighbouring CTAs read neighbouring parts of the same rows.
  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    const int c0 = (w % nstrips) * kColStrip, kb = w / nstrips;
    __syncthreads();  // the previous block is consumed (and the table is built)
    {
      // Thread t stages column c = t % 64, rows i0 + 8 j (i0 = t / 64): each
      // warp loads 32 consecutive elements of a row.  Element e of the
      // column's 8-element group g sits at slot (e + g/2) mod 8 of the group,
      // so that the 16 threads of a column, reading element e of their
      // groups at once, hit 16 distinct bank pairs.
      static_assert(kColThreads == 8 * kColStrip, "eight rows of the strip per pass");
      const int c = threadIdx.x % kColStrip, i0 = threadIdx.x / kColStrip;
      const int cc = c0 + c, row0 = kb * 128 + i0;
      const double* src = X + static_cast<long long>(row0) * ldx + cc;
      const long long step = 8 * ldx;
      double* dst = tile + c * kColPitchF64;
      double v[16];
      if (cc < cols && kb * 128 + 128 <= k) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = src[j * step];
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = (cc < cols && row0 + 8 * j < k) ? src[j * step] : 0.0;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[(j << 3) + ((i0 + (j >> 1)) & 7)] = v[j];
    }
    __syncthreads();
#pragma unroll 1
    for (int half = 0; half < 2; ++half) {
      const int c = half * 32 + cl;
      const int gcol = c0 + c;
      const unsigned long long mx = gcol < cols ? colmax[gcol] : 0ull;
      const int s = mx ? p - frexp_exp_bits(mx) : 0;
      if (kb == 0 && wd == 0 && gcol < cols) {
        shifts[gcol] = s;
        if (mx >= 0x7FF0000000000000ull) atomicOr(flags, kFlagNonFinite);
      }
      uint32_t* o = reinterpret_cast<uint32_t*>(planes + static_cast<long long>(gcol) * row_bytes + kb * kRun) + wd;
      uint32_t* o2 = NL == 1 ? reinterpret_cast<uint32_t*>(planes + kSingle * modulus_stride +
                                                           static_cast<long long>(gcol) * row_bytes2 + kb * 128) +
                                   wd
                             : nullptr;
      const double* src = tile + c * kColPitchF64 + 8 * wd;
      // The fast rounding needs the column's largest magnitude normal
      // (p <= 52); taken when every column of the warp allows it.
      const bool fast = (mx >> 52) != 0 && p <= 52;
      if (__all_sync(0xFFFFFFFFu, fast))
        col_words<R, NL, true>(src, wd >> 1, s, tb, lane_hi, o, modulus_stride / 4, o2, modulus_stride2 / 4);
      else
        col_words<R, NL, false>(src, wd >> 1, s, tb, lane_hi, o, modulus_stride / 4, o2, modulus_stride2 / 4);
    }
  }
}

int split_grid(int rows_p) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int g = sms * kSplitBlocksPerSM;  // resident CTAs per SM (registers and shared memory)
  return rows_p < g ? rows_p : g;
}

}  // namespace

template <int R, bool kRes8, int NL>
cudaError_t launch_split_r(const double* X, long long ldx, int rows, int k, int p, uint8_t* planes, int32_t* shifts,
                           uint32_t* flags, cudaStream_t stream) {
  const int rows_p = round_up(rows, kRowAlign), k_p = round_up(k, kKAlign);
  const size_t smem = static_cast<size_t>(kTableWords + 256) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(split_rows_f64_kernel<R, kRes8, NL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  split_rows_f64_kernel<R, kRes8, NL><<<split_grid(rows_p), kSplitThreads, smem, stream>>>(X, ldx, rows, k, rows_p, k_p,
                                                                                       p, planes, shifts, flags);
  return cudaGetLastError();
}

// Two-limb moduli only for FP4 planes (the INT8 comparison path takes the
// 3-limb list).
template <int R, bool kRes8>
cudaError_t launch_split_limbs(const double* X, long long ldx, int rows, int k, int p, int limbs, uint8_t* planes,
                               int32_t* shifts, uint32_t* flags, cudaStream_t stream) {
  if (limbs == 3) return launch_split_r<R, kRes8, 3>(X, ldx, rows, k, p, planes, shifts, flags, stream);
  if constexpr (!kRes8) {
    if (limbs == 2) return launch_split_r<R, false, 2>(X, ldx, rows, k, p, planes, shifts, flags, stream);
  }
  return cudaErrorInvalidValue;
}

template <bool kRes8>
cudaError_t launch_split_mode(const double* X, long long ldx, int rows, int k, int p, const SplitModuli& mods,
                              uint8_t* planes, int32_t* shifts, uint32_t* flags, cudaStream_t stream) {
  if (mods.limbs == 1) {  // the mixed-digit list (FP4 planes only), r up to kMaxModuliMix
    if constexpr (kRes8) {
      return cudaErrorInvalidValue;
    } else {
      switch (mods.r) {
#define OZEMU_SPLIT_MIX(R) \
  case R:                  \
    return launch_split_r<R, false, 1>(X, ldx, rows, k, p, planes, shifts, flags, stream);
        OZEMU_SPLIT_MIX(1) OZEMU_SPLIT_MIX(2) OZEMU_SPLIT_MIX(3) OZEMU_SPLIT_MIX(4) OZEMU_SPLIT_MIX(5)
        OZEMU_SPLIT_MIX(6) OZEMU_SPLIT_MIX(7) OZEMU_SPLIT_MIX(8) OZEMU_SPLIT_MIX(9) OZEMU_SPLIT_MIX(10)
        OZEMU_SPLIT_MIX(11) OZEMU_SPLIT_MIX(12) OZEMU_SPLIT_MIX(13) OZEMU_SPLIT_MIX(14) OZEMU_SPLIT_MIX(15)
        OZEMU_SPLIT_MIX(16) OZEMU_SPLIT_MIX(17) OZEMU_SPLIT_MIX(18) OZEMU_SPLIT_MIX(19) OZEMU_SPLIT_MIX(20)
#undef OZEMU_SPLIT_MIX
        default:
          return cudaErrorInvalidValue;
      }
    }
  }
  switch (mods.r) {
#define OZEMU_SPLIT_CASE(R) \
  case R:                   \
    return launch_split_limbs<R, kRes8>(X, ldx, rows, k, p, mods.limbs, planes, shifts, flags, stream);
    OZEMU_SPLIT_CASE(1) OZEMU_SPLIT_CASE(2) OZEMU_SPLIT_CASE(3) OZEMU_SPLIT_CASE(4) OZEMU_SPLIT_CASE(5)
    OZEMU_SPLIT_CASE(6) OZEMU_SPLIT_CASE(7) OZEMU_SPLIT_CASE(8) OZEMU_SPLIT_CASE(9) OZEMU_SPLIT_CASE(10)
    OZEMU_SPLIT_CASE(11) OZEMU_SPLIT_CASE(12) OZEMU_SPLIT_CASE(13) OZEMU_SPLIT_CASE(14) OZEMU_SPLIT_CASE(15)
    OZEMU_SPLIT_CASE(16)
#undef OZEMU_SPLIT_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

template <int R, int NL>
cudaError_t launch_split_cols_r(const double* X, long long ldx, int k, int cols, int p, uint8_t* planes,
                                int32_t* shifts, unsigned long long* colmax, uint32_t* flags, cudaStream_t stream) {
  const int cols_p = round_up(cols, kRowAlign), k_p = round_up(k, kKAlign);
  cudaError_t e = cudaMemsetAsync(colmax, 0, static_cast<size_t>(cols) * sizeof(unsigned long long), stream);
  if (e != cudaSuccess) return e;
  if (k > 0) {
    dim3 g1((cols + kColStrip - 1) / kColStrip, (k + kColMaxRows - 1) / kColMaxRows);
    if (g1.y > 65535) return cudaErrorInvalidValue;
    col_absmax_kernel<<<g1, 256, 0, stream>>>(X, ldx, k, cols, colmax);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t smem = static_cast<size_t>(kTableWords + 256) * sizeof(uint32_t) +
                      static_cast<size_t>(kColStrip) * kColPitchF64 * sizeof(double);
  e = cudaFuncSetAttribute(split_cols_f64_kernel<R, NL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long items = static_cast<long long>(cols_p / kColStrip) * (k_p / 128);
  const int grid = static_cast<int>(items < split_grid(1 << 30) ? items : split_grid(1 << 30));  // 2 CTAs per SM
  split_cols_f64_kernel<R, NL><<<grid, kColThreads, smem, stream>>>(X, ldx, k, cols, cols_p, k_p, p, colmax, planes,
                                                                     shifts, flags);
  return cudaGetLastError();
}

cudaError_t launch_split_cols_f64(const double* X, long long ldx, int k, int cols, int p, const SplitModuli& mods,
                                  uint8_t* planes, int32_t* shifts, unsigned long long* colmax, uint32_t* flags,
                                  cudaStream_t stream) {
  if (mods.limbs == 1) {
    switch (mods.r) {
#define OZEMU_COLS_MIX(R) \
  case R:                 \
    return launch_split_cols_r<R, 1>(X, ldx, k, cols, p, planes, shifts, colmax, flags, stream);
      OZEMU_COLS_MIX(1) OZEMU_COLS_MIX(2) OZEMU_COLS_MIX(3) OZEMU_COLS_MIX(4) OZEMU_COLS_MIX(5)
      OZEMU_COLS_MIX(6) OZEMU_COLS_MIX(7) OZEMU_COLS_MIX(8) OZEMU_COLS_MIX(9) OZEMU_COLS_MIX(10)
      OZEMU_COLS_MIX(11) OZEMU_COLS_MIX(12) OZEMU_COLS_MIX(13) OZEMU_COLS_MIX(14) OZEMU_COLS_MIX(15)
      OZEMU_COLS_MIX(16) OZEMU_COLS_MIX(17) OZEMU_COLS_MIX(18) OZEMU_COLS_MIX(19) OZEMU_COLS_MIX(20)
#undef OZEMU_COLS_MIX
      default:
        return cudaErrorInvalidValue;
    }
  }
  switch (mods.r) {
#define OZEMU_COLS_CASE(R)                                                                                     \
  case R:                                                                                                      \
    if (mods.limbs == 3) return launch_split_cols_r<R, 3>(X, ldx, k, cols, p, planes, shifts, colmax, flags, stream); \
    if (mods.limbs == 2) return launch_split_cols_r<R, 2>(X, ldx, k, cols, p, planes, shifts, colmax, flags, stream); \
    return cudaErrorInvalidValue;
    OZEMU_COLS_CASE(1) OZEMU_COLS_CASE(2) OZEMU_COLS_CASE(3) OZEMU_COLS_CASE(4) OZEMU_COLS_CASE(5)
    OZEMU_COLS_CASE(6) OZEMU_COLS_CASE(7) OZEMU_COLS_CASE(8) OZEMU_COLS_CASE(9) OZEMU_COLS_CASE(10)
    OZEMU_COLS_CASE(11) OZEMU_COLS_CASE(12) OZEMU_COLS_CASE(13) OZEMU_COLS_CASE(14) OZEMU_COLS_CASE(15)
    OZEMU_COLS_CASE(16)
#undef OZEMU_COLS_CASE
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

cudaError_t launch_split_cols_s8(const int8_t* X, long long ldx, int k, int cols, uint8_t* planes,
                                 cudaStream_t stream) {
  const int cols_p = round_up(cols, kRowAlign), k_p = round_up(k, kKAlign);
  if (k_p / 128 > 65535) return cudaErrorInvalidValue;  // grid.y limit
  dim3 grid(cols_p / kColTile, k_p / 128);
  split_cols_s8_kernel<<<grid, 256, 0, stream>>>(X, ldx, k, cols, k_p, planes);
  return cudaGetLastError();
}

cudaError_t launch_split_rows_four(const int8_t* X, long long ldx, int rows, int k, const FourCodes& codes,
                                   uint8_t* planes, uint32_t* flags, cudaStream_t stream) {
  const int rows_p = round_up(rows, kRowAlign), k_p = round_up(k, kKAlign);
  split_rows_four_kernel<<<split_grid(rows_p), kSplitThreads, 0, stream>>>(X, ldx, rows, k, rows_p, k_p, planes,
                                                                           codes, flags);
  return cudaGetLastError();
}

cudaError_t launch_split_cols_four(const int8_t* X, long long ldx, int k, int cols, const FourCodes& codes,
                                   uint8_t* planes, uint32_t* flags, cudaStream_t stream) {
  const int cols_p = round_up(cols, kRowAlign), k_p = round_up(k, kKAlign);
  if (k_p / 128 > 65535) return cudaErrorInvalidValue;  // grid.y limit
  dim3 grid(cols_p / 64, k_p / 128);
  split_cols_four_kernel<<<grid, 256, 0, stream>>>(X, ldx, k, cols, k_p, planes, codes, flags);
  return cudaGetLastError();
}

cudaError_t launch_transpose_f64(const double* in, long long ldin, int rows, int cols, double* out,
                                 long long ldout, cudaStream_t stream) {
  dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
  transpose_kernel<double><<<grid, block, 0, stream>>>(in, ldin, rows, cols, out, ldout);
  return cudaGetLastError();
}

}  // namespace ozemu
