// Host-side launchers of the ozemu kernels (internal to libozemu.so).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"

namespace ozemu {

inline int round_up(int x, int a) { return (x + a - 1) / a * a; }

// Deconstruction of the rows of X into limb planes (split.cu).
cudaError_t launch_split_rows_f64(const double* X, long long ldx, int rows, int k, int p, const SplitModuli& mods,
                                  uint8_t* planes, int32_t* shifts, uint32_t* flags, cudaStream_t stream);
cudaError_t launch_split_rows_f64_res8(const double* X, long long ldx, int rows, int k, int p,
                                       const SplitModuli& mods, int8_t* res8, int32_t* shifts, uint32_t* flags,
                                       cudaStream_t stream);
cudaError_t launch_split_rows_s8(const int8_t* X, long long ldx, int rows, int k, uint8_t* planes,
                                 cudaStream_t stream);
// Deconstruction of the columns of X (k x cols, row-major) into limb planes
// (plane row j = column j) without a transposed copy: a column-maximum pass
// into colmax (cols words of device scratch, zeroed here), then the split.
cudaError_t launch_split_cols_f64(const double* X, long long ldx, int k, int cols, int p, const SplitModuli& mods,
                                  uint8_t* planes, int32_t* shifts, unsigned long long* colmax, uint32_t* flags,
                                  cudaStream_t stream);
// The four planes of INT8-stored operands for the INT4 x INT8 product
// (rows of A; columns of B, k >= 1), layout [rows_p][k_p/128][4][64];
// values the code table marks out of range raise kFlagRange.
cudaError_t launch_split_rows_four(const int8_t* X, long long ldx, int rows, int k, const FourCodes& codes,
                                   uint8_t* planes, uint32_t* flags, cudaStream_t stream);
cudaError_t launch_split_cols_four(const int8_t* X, long long ldx, int k, int cols, const FourCodes& codes,
                                   uint8_t* planes, uint32_t* flags, cudaStream_t stream);
cudaError_t launch_transpose_f64(const double* in, long long ldin, int rows, int cols, double* out,
                                 long long ldout, cudaStream_t stream);
// INT8 limb planes of the columns of X (k x cols, row-major, k >= 1): plane
// row j holds column j.
cudaError_t launch_split_cols_s8(const int8_t* X, long long ldx, int k, int cols, uint8_t* planes,
                                 cudaStream_t stream);

// FP4 limb GEMM (gemm_fp4.cu).  Residue mode writes uint8 [r][m][ldr]
// residues; int mode (r = 1) writes int32 C32 with leading dimension ldc.
// kc_blocks: 128-wide K blocks per exactly accumulated chunk.
struct LimbGemmCall {
  bool residue_mode;
  int m, n, k, r;
  const uint8_t* a_planes;
  const uint8_t* b_planes;
  uint8_t* res_out;
  long long ldr;
  int32_t* c32;
  long long ldc;
  int kc_blocks;
  // Digit planes per modulus: 3 (three-limb moduli, or the INT8 product), 2
  // (two-limb moduli) or 1 (single-digit moduli), residue mode; 4: the four
  // planes of the INT4 x INT8 product (int mode, r = 1, any K).
  int limbs = 3;
  EpiModuli em;
  uint32_t* flags;
};
cudaError_t launch_limb_gemm(const LimbGemmCall& call, cudaStream_t stream);

// INT8 residue GEMM with legacy mma.sync (igemm_mma.cu): the comparison
// variant computing each modulus's residue product in one INT8 GEMM.
cudaError_t launch_residue_gemm_i8(int m, int n, int k, int r, const int8_t* a_res8, const int8_t* b_res8,
                                   uint8_t* res_out, long long ldr, const EpiModuli& em, cudaStream_t stream);

// Fused deconstruction + product for narrow B (gemv.cu): residues of
// C = A B for n <= kNarrowMaxN columns without limb planes.  Writes the
// residues [r][m][ldr] and shifts that launch_crt_f64 consumes.
// Output columns of one CTA-pair limb-GEMM tile (gemm_fp4.cu).
constexpr int kPairTileCols = 224;

constexpr int kNarrowMaxN = 2;
constexpr int kNarrowMaxK = 1 << 24;
constexpr int kNarrowMaxP = 52;  // p_A: scaled elements are right shifts of the significand
struct NarrowCall {
  int m, n, k, kp;  // kp: k rounded up to 16
  int pA, pB;
  const double* A;
  long long lda;
  const double* B;
  long long ldb;
  NarrowModuli nm;
  uint8_t* bres;    // [n][r][kp] residues of B's columns
  int32_t* colsum;  // [n][r] sum_k b mod m
  uint8_t* res;     // [r][m][ldr]
  long long ldr;
  int32_t* sa;
  int32_t* sb;
  uint32_t* flags;
};
cudaError_t launch_narrow_residues(const NarrowCall& call, cudaStream_t stream);

// CRT and scale back (crt.cu).
cudaError_t launch_crt_f64(int m, int n, const uint8_t* residues, long long ldr, const int32_t* sa,
                           const int32_t* sb, double* C, long long ldc, const CrtModuli& cm, cudaStream_t stream);

// Fill helpers.
cudaError_t launch_zero_f64(double* C, int m, int n, long long ldc, cudaStream_t stream);
cudaError_t launch_zero_s32(int32_t* C, int m, int n, long long ldc, cudaStream_t stream);

}  // namespace ozemu
