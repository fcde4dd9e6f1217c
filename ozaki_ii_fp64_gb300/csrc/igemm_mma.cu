// INT8 residue GEMM for comparison: each modulus's residue product computed
// directly as one INT8 x INT8 -> INT32 GEMM (instead of 9 FP4 limb GEMMs),
// then reduced modulo m_l.
//
// The tcgen05 INT8 kind is not available on sm_103a (ptxas rejects
// `kind::i8` for this target), so this variant uses the legacy warp-level
// mma.sync.m16n8k32 s8 tensor instruction: 128 x 128 CTA tiles, 8 warps of
// 64 x 32, a 3-stage cp.async pipeline over 128-byte K slices held in
// shared memory with a 16-byte-chunk XOR swizzle (conflict-free ldmatrix).
//
// Inputs are the balanced int8 residues written by the res8 split:
// a_res8 [r][round_up(m,128)][round_up(k,128)], b_res8 likewise for the
// columns of B.  Output: the residue layout of the FP4 path, [r][m][ldr].
// Exact while |sum| < 2^31, i.e. k <= 131071 for int8 residues.
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kTile = 128;
constexpr int kBK = 128;                     // bytes (= int8 elements) of K per stage
constexpr int kStagesI8 = 3;
constexpr int kStageBytes = 2 * kTile * kBK; // A and B slices
constexpr int kThreadsI8 = 256;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * kBK + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t saddr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(saddr)
               : "memory");
}

__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct I8Args {
  int m, n, kb_total;
  int rows_a_p, rows_b_p, k_p;
  int tiles_m, tiles_n;
  const int8_t* a;
  const int8_t* b;
  uint8_t* res_out;
  long long ldr;
  EpiModuli em;
};

__global__ void __launch_bounds__(kThreadsI8) residue_gemm_i8_kernel(const I8Args args) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int per_mod = args.tiles_m * args.tiles_n;
  const int l = blockIdx.x / per_mod;
  const int t = blockIdx.x % per_mod;
  const int tm = t % args.tiles_m, tn = t / args.tiles_m;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp & 1, wn = warp >> 1;  // 2 x 4 warps of 64 x 32

  const int8_t* a_base = args.a + (static_cast<long long>(l) * args.rows_a_p + tm * kTile) * args.k_p;
  const int8_t* b_base = args.b + (static_cast<long long>(l) * args.rows_b_p + tn * kTile) * args.k_p;
  const uint32_t s0 = smem_u32(smem);

  auto load_stage = [&](int kb, int stage) {
    const uint32_t sa = s0 + stage * kStageBytes, sb = sa + kTile * kBK;
#pragma unroll
    for (int i = 0; i < (kTile * kBK / 16) / kThreadsI8; ++i) {
      const int idx = threadIdx.x + i * kThreadsI8;  // 0 .. 1023
      const int row = idx >> 3, chunk = idx & 7;
      const long long goff = static_cast<long long>(row) * args.k_p + kb * kBK + chunk * 16;
      cp_async16(sa + swz(row, chunk), a_base + goff);
      cp_async16(sb + swz(row, chunk), b_base + goff);
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][j][q] = 0;

  const int kb_total = args.kb_total;
#pragma unroll
  for (int s = 0; s < kStagesI8 - 1; ++s) {
    if (s < kb_total) load_stage(s, s);
    cp_async_commit();
  }
  for (int kb = 0; kb < kb_total; ++kb) {
    cp_async_wait<kStagesI8 - 2>();
    __syncthreads();
    const int nxt = kb + kStagesI8 - 1;
    if (nxt < kb_total) load_stage(nxt, nxt % kStagesI8);
    cp_async_commit();
    const uint32_t sa = s0 + (kb % kStagesI8) * kStageBytes, sb = sa + kTile * kBK;
#pragma unroll
    for (int kk = 0; kk < kBK / 32; ++kk) {
      uint32_t af[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = wm * 64 + i * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int chunk = 2 * kk + (lane >> 4);
        ldmatrix_x4(sa + swz(row, chunk), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
      uint32_t bf[4][2];
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const int row = wn * 32 + j * 8 + (lane & 7) + (lane >> 4) * 8;
        const int chunk = 2 * kk + ((lane >> 3) & 1);
        ldmatrix_x4(sb + swz(row, chunk), bf[j][0], bf[j][1], bf[j + 1][0], bf[j + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_s8(acc[i][j], af[i], bf[j][0], bf[j][1]);
    }
  }
  cp_async_wait<0>();

  // Epilogue: residues modulo m_l in [0, m_l).
  const int ml = static_cast<int>(args.em.m[l]);
  const int g = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = tm * kTile + wm * 64 + i * 16 + g + h * 8;
      if (row >= args.m) continue;
      uint8_t* rrow = args.res_out + (static_cast<long long>(l) * args.m + row) * args.ldr;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = tn * kTile + wn * 32 + j * 8 + tq * 2;
        if (col >= args.ldr) continue;
        int v0 = acc[i][j][2 * h] % ml, v1 = acc[i][j][2 * h + 1] % ml;
        v0 += v0 < 0 ? ml : 0;
        v1 += v1 < 0 ? ml : 0;
        *reinterpret_cast<uint16_t*>(rrow + col) = static_cast<uint16_t>(v0 | (v1 << 8));
      }
    }
  }
}

}  // namespace

cudaError_t launch_residue_gemm_i8(int m, int n, int k, int r, const int8_t* a_res8, const int8_t* b_res8,
                                   uint8_t* res_out, long long ldr, const EpiModuli& em, cudaStream_t stream) {
  I8Args a;
  a.m = m;
  a.n = n;
  a.k_p = round_up(k, kKAlign);
  a.kb_total = a.k_p / kBK;
  a.rows_a_p = round_up(m, kRowAlign);
  a.rows_b_p = round_up(n, kRowAlign);
  a.tiles_m = a.rows_a_p / kTile;
  a.tiles_n = a.rows_b_p / kTile;
  a.a = a_res8;
  a.b = b_res8;
  a.res_out = res_out;
  a.ldr = ldr;
  a.em = em;
  const int smem = kStagesI8 * kStageBytes;
  cudaError_t e = cudaFuncSetAttribute(residue_gemm_i8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(r) * a.tiles_m * a.tiles_n;
  residue_gemm_i8_kernel<<<static_cast<unsigned>(grid), kThreadsI8, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ozemu
