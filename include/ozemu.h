/*
 * ozemu -- Ozaki scheme II FP64 emulation on GB300 (sm_103a) FP4 tensor cores.
 *
 * C ABI of libozemu.so.  Plain pointers and sizes only.  Unless a comment
 * says "host", every pointer argument is a DEVICE pointer owned by the
 * caller, and every call only enqueues work on `stream` and returns without
 * synchronising (ozemu_get_status is the one call that synchronises).
 *
 * Sources the operations follow (cited by page title and section):
 *   [TME4] "The Missing Fourth Term for the Emulation Tensor Memory
 *          Equilibrium (TME) Model: The Residue Deconstruction Cost"
 *          (arXiv 2610.10924), abstract -- Ozaki scheme II: each fp64 row/column
 *          is scaled by a power of two, rounded to an integer and reduced
 *          modulo each of r moduli; per-output reconstruction.
 *   [AWE]  arXiv 2609.24519 (Adaptive Weight Encoding for FP4 tensor cores),
 *          English abstract -- digits in S = {0,+-1,+-2,+-3,+-4,+-6,+-8,+-12}
 *          (FP4 e2m1 values times two), base-13 limbs with weights
 *          (1, 13, 169), 9 exact FP4 GEMMs per INT8 x INT8 product, 4 per
 *          INT4 x INT8 product, the same formulation modulo m.
 *
 * Conventions
 *   - Matrices are row-major.  A is m x k (leading dimension lda >= k),
 *     B is k x n (ldb >= n), C is m x n (ldc >= n).  C = A B, no alpha/beta.
 *   - Moduli: the greedy pairwise-coprime integers counting down from 256
 *     (256, 255, 253, 251, 247, 241, ...); r of them, 1 <= r <= ozemu_max_moduli().
 *   - Bit budget for inner dimension k: P is the largest integer with
 *     2 k 2^P < m_1 m_2 ... m_r; p_A = ceil(P/2), p_B = floor(P/2).
 *   - Row shift s_i = p - e_i, where e_i is the frexp exponent of the row's
 *     largest magnitude (2^(e_i-1) <= max < 2^e_i); 0 for an all-zero row.
 *     Integers are round-half-to-even(x 2^s).
 *   - Residues are balanced: in [-floor(m/2), ceil(m/2) - 1] (int8 range).
 *   - Limb split of a residue x: x = d0 + 13 d1 + 169 d2 with d_i in S; the
 *     low digits are the smallest-magnitude member of S in x's class mod 13.
 *
 * Limb-plane layout (written by the split calls, read by the GEMM calls)
 *   rows_p = round_up(rows, 128), k_p = round_up(k, 128), row_bytes =
 *   3 k_p/2.  Row i of modulus l (0-based) starts at byte
 *   (l*rows_p + i) * row_bytes.  A row holds, for each 128-element K block
 *   kb, the 64 bytes of limb 0, then of limb 1, then of limb 2: limb j of
 *   element k is at row byte (3*(k/128) + j)*64 + (k%128)/2, the 4-bit FP4
 *   e2m1 code of d_j/2, low nibble for even k.  Padding rows and columns hold
 *   digit 0 (code 0).  INT8 planes are the same with a single "modulus".
 *   Total bytes: ozemu_plane_bytes(rows, k, r).
 *
 * Residue layout (written by ozemu_residue_gemm, read by ozemu_crt_f64)
 *   uint8 [r][m][ldr], ldr = round_up(n, 16): residue of C' modulo m_l in
 *   [0, m_l) at byte (l*m + i)*ldr + j.  Total bytes: ozemu_residue_bytes.
 *
 * Concurrency: the workspace is cached per device and shared by the calls
 * that use it, so calls on one device must not overlap in time on different
 * streams (issue them on one stream, or synchronise in between).
 *
 * Errors: calls return an ozemu_status.  Argument checks happen on the host
 * before anything is enqueued.  Device-side conditions (non-finite input,
 * an INT4 value outside [-8, 7], a pipeline wait that hit its time limit)
 * set a per-device flag that ozemu_get_status reports and clears.
 */
#ifndef OZEMU_H
#define OZEMU_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OZEMU_OK = 0,
  OZEMU_ERR_INVALID_ARG = -1, /* bad size, pointer, leading dim, r or p      */
  OZEMU_ERR_K_OVERFLOW = -2,  /* int32 result could overflow (k > 131071)   */
  OZEMU_ERR_ALLOC = -3,       /* workspace allocation failed                */
  OZEMU_ERR_CUDA = -4,        /* a CUDA call or launch failed               */
  OZEMU_ERR_NONFINITE = -5,   /* an input held Inf or NaN (output unspecified) */
  OZEMU_ERR_TIMEOUT = -6,     /* a kernel pipeline wait hit its time limit  */
  OZEMU_ERR_UNSUPPORTED = -7, /* current device is not sm_103 (GB300)       */
  OZEMU_ERR_SCRATCH_TOO_SMALL = -8, /* problem needs more than the fixed scratch */
  OZEMU_ERR_RANGE = -9        /* an INT4 operand held a value outside [-8, 7] */
} ozemu_status;

/* ------------------------------------------------------------------------ */
/* Full products                                                             */
/* ------------------------------------------------------------------------ */

/* Exact C32 = A B for int8 A (m x k, row-major, lda = k) and int8 B (k x n,
 * row-major, ldb = n); C32 int32 m x n row-major (ldc = n).  Each operand is
 * split into 3 base-13 limbs and the product takes 9 FP4 GEMMs, recombined
 * with weights 13^(i+j) ([AWE] abstract).  k > 131071 -> OZEMU_ERR_K_OVERFLOW.
 * m, n or k = 0 is a no-op (k = 0 zeroes C32).  Uses the cached workspace. */
int ozemu_igemm_s8(int m, int n, int k, const int8_t* A, const int8_t* B,
                   int32_t* C32, cudaStream_t stream);

/* Exact C32 = A B for INT4 A (m x k, values in [-8, 7] stored one per int8,
 * row-major, lda = k) and int8 B (k x n, row-major, ldb = n); C32 int32
 * m x n row-major (ldc = n).  [AWE] abstract: an INT4 x INT8 product in four
 * FP4 products.  Encoding: a b = sum_k g_k u_k(a) v_k(b) with g = (3, 2, 6,
 * 12) and every plane value in S = {0, +-1, +-2, +-3, +-4, +-6, +-8, +-12};
 * the B planes lie on the relation sum_k t_k g_k v_k = 0, t = (-12, -9, -6,
 * 3/2), and u_k(a) = a + t_k z(a).  The four plane products go into one fp32
 * accumulator per tile (the weights carried by the block scales), exact over
 * K chunks of 8192 (|running value| <= 1024 per K element), summed in int32.
 * An element of A outside [-8, 7] counts as 0 and makes the next
 * ozemu_get_status() return OZEMU_ERR_RANGE.  k > 2097151 ->
 * OZEMU_ERR_K_OVERFLOW; m, n or k = 0 is a no-op (k = 0 zeroes C32).  Uses
 * the cached workspace.  device pointers; stream-ordered. */
int ozemu_igemm_s4s8(int m, int n, int k, const int8_t* A, const int8_t* B, int32_t* C32, cudaStream_t stream);

/* Emulated fp64 C = A B with r moduli: deconstruction of A's rows and B's
 * columns ([TME4] abstract), 9 FP4 limb GEMMs per modulus with modular
 * recombination ([AWE] abstract), CRT and one correct rounding per entry of
 * C' 2^-(s_i + t_j).  Requires 2k < m_1...m_r (else OZEMU_ERR_INVALID_ARG).
 * m, n or k = 0 is a no-op (k = 0 zeroes C).  Inf/NaN in A or B sets the
 * non-finite flag; C is then unspecified.  Uses the cached workspace.
 * For n <= ozemu_narrow_max_n(), k <= 2^24 and p_A <= 52 (every k when
 * r <= 13) the residues come from the fused narrow path
 * (ozemu_residues_narrow_f64) instead of limb planes; the result is the same
 * bit for bit. */
int ozemu_dgemm(int m, int n, int k, const double* A, int lda, const double* B,
                int ldb, double* C, int ldc, int r, cudaStream_t stream);

/* ozemu_dgemm with HOST buffers: A (m x k, lda), B (k x n, ldb) and C
 * (m x n, ldc) are row-major host pointers; the result is the same as
 * ozemu_dgemm's, bit for bit.  The copies in and out are pipelined with the
 * work: column blocks of B and row chunks of A are copied on a copy stream
 * while earlier blocks and chunks are deconstructed and multiplied on
 * `stream`; each (chunk, block) product's CRT runs on a second stream beside
 * the next product, and each finished block of C is copied out at once.  Page-locked (pinned) host buffers are needed for
 * the copies to overlap; pageable ones give the same result, serialised.
 * All work is ordered after what `stream` already holds, and `stream`
 * completes only after C is on the host: synchronise `stream` (or call
 * ozemu_get_status on it) before reading C.  The source pages have no
 * counterpart; this is the end-to-end entry point.  Errors as ozemu_dgemm.
 * Uses the cached workspace (it also holds device copies of A, B and C). */
int ozemu_dgemm_host(int m, int n, int k, const double* A, int lda, const double* B,
                     int ldb, double* C, int ldc, int r, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Host-side queries (no device work)                                       */
/* ------------------------------------------------------------------------ */

/* Largest supported r (16: keeps p_A, p_B <= 62 for every k >= 1). host. */
int ozemu_max_moduli(void);

/* Writes the first r moduli to out[0..r-1] (host pointer). host. */
int ozemu_moduli(int r, int32_t* out);

/* Bit budget for inner dimension k and r moduli: *p_a = ceil(P/2),
 * *p_b = floor(P/2) (host pointers).  OZEMU_ERR_INVALID_ARG if 2k >= M. host. */
int ozemu_bit_budget(int k, int r, int* p_a, int* p_b);

/* Bytes of the limb planes of `rows` rows of length k with r moduli
 * (r = 1 for INT8 planes); 0 on bad arguments.  host. */
size_t ozemu_plane_bytes(int rows, int k, int r);

/* Bytes of the residue output of an m x n product with r moduli (r up to
 * 20, the mixed-digit list's limit; 0 on bad arguments). host. */
size_t ozemu_residue_bytes(int m, int n, int r);

/* ------------------------------------------------------------------------ */
/* Stages (stored limb planes / residues can be reused across products)     */
/* ------------------------------------------------------------------------ */

/* Deconstruct the rows of X (rows x k, row-major, ldx >= k) with budget p
 * (0 <= p <= 62, from ozemu_bit_budget) and r moduli: writes shifts[rows]
 * (int32, s_i) and the limb planes (ozemu_plane_bytes(rows, k, r) bytes).
 * [TME4] abstract (scale, round, reduce); [AWE] abstract (limbs in S). */
int ozemu_split_rows_f64(int rows, int k, const double* X, int ldx, int p, int r,
                         uint8_t* planes, int32_t* shifts, cudaStream_t stream);

/* Same for the columns of X (k x cols, row-major, ldx >= cols): column j
 * becomes plane row j.  Two passes over X, no transposed copy: the column
 * maxima (the cached workspace holds them, 8 bytes per column), then the
 * split of 128-row x 64-column blocks staged in shared memory. */
int ozemu_split_cols_f64(int k, int cols, const double* X, int ldx, int p, int r,
                         uint8_t* planes, int32_t* shifts, cudaStream_t stream);

/* Four-plane layout of the INT4 x INT8 product: uint8
 * [rows_p][k_p/128][4][64], for each 128-element K block the 64 bytes of
 * each of the four planes (two FP4 e2m1 codes of digit / 2 per byte, low
 * nibble = even k); rows_p = rows rounded up to 128, k_p = k rounded up to
 * 128, padding digit 0.  Bytes for rows x k; 0 on negative sizes. */
size_t ozemu_four_plane_bytes(int rows, int k);

/* The four planes u_k of the rows of an INT4 matrix X (rows x k, values in
 * [-8, 7] one per int8, leading dimension ldx >= k), for
 * ozemu_igemm_s4s8's encoding; out-of-range values as there.  planes: device,
 * 16-byte aligned, ozemu_four_plane_bytes(rows, k) bytes. */
int ozemu_split_rows_s4(int rows, int k, const int8_t* X, int ldx, uint8_t* planes, cudaStream_t stream);

/* The four planes v_k of the columns of an int8 matrix X (k x cols,
 * row-major, leading dimension ldx >= cols): plane row j holds column j. */
int ozemu_split_cols_s8_four(int k, int cols, const int8_t* X, int ldx, uint8_t* planes, cudaStream_t stream);

/* INT8 limb planes of the rows of X (rows x k, ldx >= k): 3 planes. */
int ozemu_split_rows_s8(int rows, int k, const int8_t* X, int ldx,
                        uint8_t* planes, cudaStream_t stream);

/* INT8 limb planes of the columns of X (k x cols, ldx >= cols). Workspace. */
int ozemu_split_cols_s8(int k, int cols, const int8_t* X, int ldx,
                        uint8_t* planes, cudaStream_t stream);

/* Residues of C' = A'B' modulo each of r moduli, from limb planes of A's rows
 * (m rows) and B's columns (n rows), inner dimension k: 9 FP4 GEMMs per
 * modulus, recombined modulo m_l ([AWE] abstract: the formulation holds
 * modulo m).  Output in the residue layout above. */
int ozemu_residue_gemm(int m, int n, int k, int r, const uint8_t* a_planes,
                       const uint8_t* b_planes, uint8_t* residues, cudaStream_t stream);

/* Exact int32 C32 = sum_{i,j} 13^(i+j) A_i B_j from INT8 limb planes
 * ([AWE] abstract); C32 m x n row-major with leading dimension ldc >= n.
 * k > 131071 -> OZEMU_ERR_K_OVERFLOW. */
int ozemu_limb_gemm_s32(int m, int n, int k, const uint8_t* a_planes,
                        const uint8_t* b_planes, int32_t* C32, int ldc,
                        cudaStream_t stream);

/* Largest n taken by ozemu_residues_narrow_f64 (2). host. */
int ozemu_narrow_max_n(void);

/* Residues of C' = A'B' for a narrow product, 1 <= n <= ozemu_narrow_max_n()
 * and 1 <= k <= 2^24, without limb planes: the deconstruction of A's rows is
 * fused with the products.  [TME4] abstract: below the critical intensity
 * OI* the deconstruction of the streamed operand (the fourth term of the TME
 * model) bounds the emulation, so each element of A is read once, scaled,
 * rounded and reduced modulo every m_l in registers and multiplied with B's
 * residues at once; the modular reduction of the sums happens once per
 * output.  A (m x k, lda >= k) and B (k x n, ldb >= n) are row-major fp64
 * device pointers.  Writes shifts_a[m] and shifts_b[n] (int32, s_i and t_j
 * for the budget ozemu_bit_budget(k, r)) and the residues (residue layout
 * above, 16-byte aligned): the same bytes as ozemu_split_rows_f64 +
 * ozemu_split_cols_f64 + ozemu_residue_gemm.  Inf/NaN set the non-finite
 * flag.  Uses the cached workspace for B's residues.  n or k out of range,
 * 2k >= m_1...m_r, or a budget p_A > 52 (r >= 14 with small k) ->
 * OZEMU_ERR_INVALID_ARG. */
int ozemu_residues_narrow_f64(int m, int n, int k, int r, const double* A, int lda,
                              const double* B, int ldb, uint8_t* residues,
                              int32_t* shifts_a, int32_t* shifts_b, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* INT8 residue-GEMM comparison path                                        */
/* ------------------------------------------------------------------------ */

/* Bytes of the int8 residue planes of `rows` rows of length k, r moduli:
 * r * round_up(rows, 128) * round_up(k, 128).  0 on bad arguments. host. */
size_t ozemu_res8_bytes(int rows, int k, int r);

/* Deconstruct the rows of X like ozemu_split_rows_f64 ([TME4] abstract:
 * scale, round, reduce) but store the balanced residues themselves: int8
 * [r][round_up(rows,128)][round_up(k,128)], residue of row i, element kk of
 * modulus l at byte (l*rows_p + i)*k_p + kk; padding holds 0. */
int ozemu_split_rows_f64_res8(int rows, int k, const double* X, int ldx, int p, int r,
                              int8_t* res8, int32_t* shifts, cudaStream_t stream);

/* Same for the columns of X (k x cols, row-major).  Uses the workspace. */
int ozemu_split_cols_f64_res8(int k, int cols, const double* X, int ldx, int p, int r,
                              int8_t* res8, int32_t* shifts, cudaStream_t stream);

/* Residues of C' = A'B' modulo each modulus from int8 residue planes, one
 * INT8 x INT8 -> INT32 GEMM per modulus on the warp-level mma.sync tensor
 * path, then reduction modulo m_l.  The comparison variant of
 * ozemu_residue_gemm (same output layout and values); the tcgen05 INT8
 * kind does not exist on sm_103a.  k > 131071 -> OZEMU_ERR_K_OVERFLOW. */
int ozemu_residue_gemm_i8(int m, int n, int k, int r, const int8_t* a_res8,
                          const int8_t* b_res8, uint8_t* residues, cudaStream_t stream);

/* Per-output reconstruction ([TME4] abstract): C' in (-M/2, M/2) from its r
 * residues by the CRT in direct form, C' = sum_l c_l W_l - q M with
 * W_l = (M/m_l) ((M/m_l)^-1 mod m_l) (byte-wise integer dot products and one
 * quotient estimate q); an output whose quotient estimate is within 2^-8 of
 * ambiguous takes the exact mixed-radix (Garner) digits instead.  Then
 * C[i*ldc + j] = RN(C' 2^-(sA[i] + sB[j])), one correct rounding (subnormal
 * and overflow included). */
int ozemu_crt_f64(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a,
                  const int32_t* shifts_b, double* C, int ldc, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Status and workspace                                                      */
/* ------------------------------------------------------------------------ */

/* Synchronises `stream`, then returns and clears the current device's flags:
 * OZEMU_ERR_TIMEOUT, OZEMU_ERR_NONFINITE, OZEMU_ERR_RANGE (in that order of
 * precedence), OZEMU_ERR_CUDA (a sticky CUDA error) or OZEMU_OK.  The flags of ozemu_dgemm_noalloc are separate: see
 * ozemu_get_status_noalloc. */
int ozemu_get_status(cudaStream_t stream);

/* Frees the workspace cached for the current device (synchronises it).
 * Calls after this re-allocate on demand. */
void ozemu_release(void);

/* Caps the cached workspace of every device at `bytes` (0 removes the cap).
 * A call that needs a larger workspace then returns OZEMU_ERR_ALLOC before
 * enqueueing anything, instead of growing it; a cached block already above
 * the new cap on the current device is freed (which synchronises it).  For
 * callers that share the GPU's memory with other work.  host. */
int ozemu_set_workspace_limit(size_t bytes);

/* The cap set by ozemu_set_workspace_limit (0: none).  host. */
size_t ozemu_workspace_limit(void);

/* Diagnostic of the kernels' failure detection.  Every pipeline wait in the
 * GEMM kernels is bounded in time: a wait that gives up sets the time-out
 * flag, and the kernel drains what it issued, frees its tensor memory and
 * returns, so the context stays usable.  This call launches one CTA whose
 * thread makes the same bounded wait (limit_ns nanoseconds, 1 ns .. 1 s) on a
 * barrier phase that nothing completes, with no copy or tensor operation in
 * flight: it always gives up.  A following ozemu_get_status(stream) returns
 * OZEMU_ERR_TIMEOUT and clears the flag; until then, GEMM launches on the
 * device skip their work (they see the flag).  limit_ns out of range ->
 * OZEMU_ERR_INVALID_ARG.  The pages have no counterpart. */
int ozemu_probe_wait_timeout(unsigned long long limit_ns, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Allocation-free product                                                   */
/* ------------------------------------------------------------------------ */

/* Same result as ozemu_dgemm (bit for bit), but it never allocates device
 * memory: no cudaMalloc, cudaFree or allocating library call.  It is meant
 * for callers that cannot allocate: a host application or framework that
 * reserves the GPU's memory up front and hands out no more, code whose
 * allocation calls would synchronise the device on a latency-critical path,
 * or an environment where an allocation may fail part way through a run.
 * The source pages have no counterpart to this call; it is a packaging of
 * the same stages.
 *
 * All intermediate data (limb planes, shifts, the transposed copy of B,
 * residues and a status word) lives in one file-scope static device array of
 * 64 MiB, which every GPU that loads that part of the library holds until the
 * process exits.  The problem must fit: with rows_p(x) = round_up(x, 128),
 * k_p = round_up(k, 128) and 256-byte alignment of each part,
 *   3 r (rows_p(m) + rows_p(n)) k_p / 2 + 4 (m + n) + r m round_up(n, 16)
 *   + 8 n + 256  <=  64 MiB,
 * otherwise the call returns OZEMU_ERR_SCRATCH_TOO_SMALL before enqueueing
 * anything (for example m = n = k = 1024 with r = 13 fits; 2048^3 does not).
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array and overwrites what the last call
 * left there, so calls that overlap on the GPU (different streams, or several
 * host threads) race: serialise them.  Device-side conditions (non-finite
 * input, a pipeline wait time-out) are recorded in the array's status word,
 * which each call clears first: ozemu_get_status does not report them, and
 * ozemu_get_status_noalloc does.  After a time-out C is not the product
 * (the GEMM skipped its work and the reconstruction used stale residues), so
 * check the status before using C.  This call always takes the limb-plane
 * path, also for n <= ozemu_narrow_max_n() where ozemu_dgemm takes the fused
 * narrow path; the size formula above therefore bounds narrow shapes too
 * (m = 16384, n = 1, k = 16384 at r = 12 needs about 4.8 GB of planes and is
 * rejected).  Arguments and errors otherwise as ozemu_dgemm. */
int ozemu_dgemm_noalloc(int m, int n, int k, const double* A, int lda, const double* B,
                        int ldb, double* C, int ldc, int r, cudaStream_t stream);

/* Synchronises `stream`, then returns and clears the status word of
 * ozemu_dgemm_noalloc on the current device: OZEMU_ERR_TIMEOUT,
 * OZEMU_ERR_NONFINITE or OZEMU_OK (the word reflects the last noalloc call
 * that ran).  Allocates nothing: it copies the 4-byte word into a host
 * variable and clears it. */
int ozemu_get_status_noalloc(cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Two-limb moduli                                                          */
/* ------------------------------------------------------------------------ */

/* A variant of the same scheme with smaller moduli, so that each balanced
 * residue needs only two base-13 limbs.  [AWE] abstract: limbs in S with
 * weights (1, 13, 169) and 9 FP4 products per modulus.  Two limbs d0 + 13 d1
 * with d_i in S cover every integer of [-56, 56]: the low digit d0 is the
 * smallest-magnitude member of S in x's class mod 13 (|d0| <= 6 except for
 * classes 5 and 8, whose only members are -8 and 8), and across [-56, 56]
 * the carry d1 = (x - d0)/13 stays within [-4, 4], in S (checked for every
 * x by the oracle pins).  So a modulus m <= 113 needs no third limb.  The product of two such
 * residues then takes 4 FP4 GEMMs instead of 9:
 *   D1 = A0 B0 + 13 (A0 B1 + A1 B0),   D2 = A1 B1,   residue = D1 + 169 D2 mod m.
 * Each modulus carries about 6.7 bits instead of 8, so about 16/13 as many
 * moduli reach the same accuracy: r = 16 two-limb moduli (64 products) give
 * about the bit budget of r = 13 three-limb moduli (117 products).  The
 * pages give the three-limb form; this one is a reading of the same limb
 * algebra with the top limb fixed at zero.
 *
 *   - Moduli: the greedy pairwise-coprime integers counting down from 113
 *     (113, 112, 111, 109, 107, 103, 101, 97, 95, 89, 83, 79, 73, 71, 67, 61).
 *   - Bit budget: as above with these moduli (2k 2^P < m_1...m_r).
 *   - Limb planes: row_bytes = 2 k_p/2; a row holds, for each 128-element K
 *     block, the 64 bytes of limb 0, then of limb 1: limb j of element k is
 *     at row byte (2*(k/128) + j)*64 + (k%128)/2.  Row i of modulus l starts
 *     at byte (l*rows_p + i) * row_bytes.  Total: ozemu_plane_bytes_2limb.
 *   - Residue layout: the same as the three-limb calls, with these moduli.
 * Planes and residues of one family are not valid input to the other's
 * calls.  Arguments, ownership and errors are those of the three-limb call of
 * the same name. */
int ozemu_moduli_2limb(int r, int32_t* out);
int ozemu_bit_budget_2limb(int k, int r, int* p_a, int* p_b);
size_t ozemu_plane_bytes_2limb(int rows, int k, int r);
int ozemu_split_rows_f64_2limb(int rows, int k, const double* X, int ldx, int p, int r,
                               uint8_t* planes, int32_t* shifts, cudaStream_t stream);
int ozemu_split_cols_f64_2limb(int k, int cols, const double* X, int ldx, int p, int r,
                               uint8_t* planes, int32_t* shifts, cudaStream_t stream);
int ozemu_residue_gemm_2limb(int m, int n, int k, int r, const uint8_t* a_planes,
                             const uint8_t* b_planes, uint8_t* residues, cudaStream_t stream);
int ozemu_crt_f64_2limb(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a,
                        const int32_t* shifts_b, double* C, int ldc, cudaStream_t stream);

/* C = A B (device buffers, as ozemu_dgemm) through the two-limb stages:
 * split, 4 FP4 GEMMs per modulus, CRT, one correct rounding per entry.
 * Requires 2k < m_1...m_r of the two-limb moduli.  There is no narrow path;
 * m >= 2048 pipelines the stages over row chunks like ozemu_dgemm.  Uses the
 * cached workspace. */
int ozemu_dgemm_2limb(int m, int n, int k, const double* A, int lda, const double* B,
                      int ldb, double* C, int ldc, int r, cudaStream_t stream);

/* ozemu_dgemm_2limb with HOST buffers, pipelined like ozemu_dgemm_host (same
 * stream and synchronisation rules); the result equals ozemu_dgemm_2limb's
 * bit for bit. */
int ozemu_dgemm_host_2limb(int m, int n, int k, const double* A, int lda, const double* B,
                           int ldb, double* C, int ldc, int r, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Mixed-digit moduli: fewer FP4 products per output                        */
/* ------------------------------------------------------------------------ */

/* [AWE] abstract: the digit set S holds every residue modulo 13, encodings
 * are chosen per input range, and the formulation holds modulo m, so the
 * residue number system of Ozaki scheme II can take fewer FP4 products than
 * nine per modulus (the page counts 75 products of prior work for the FP64
 * significand and 59 with its encodings, which it does not print).  This
 * family is our reading of that: a modulus m for which S meets every residue
 * class mod m (only m <= 13: 2..9, 11, 13, found by brute force over S)
 * needs ONE digit per residue, and its residue product is ONE FP4 product.
 *
 *   - Moduli: the pairwise-coprime set of such m with the largest product,
 *     8, 13, 11, 9, 7, 5 (the "single-digit" moduli, even one first), then
 *     the greedy pairwise-coprime integers counting down from 113 coprime to
 *     those (113, 109, 107, 103, 101, 97, 89, 83, 79, 73, 71, 67, 61, 59),
 *     which take two base-13 digits and 4 FP4 products as the two-limb
 *     moduli do.  1 <= r <= ozemu_max_moduli_mixed() (20).
 *   - Digits: for a single-digit modulus, the balanced residue x itself when
 *     it lies in S, else the member of S in x's class of smallest magnitude
 *     (13: +-5 -> -+8; 11: +-5 -> -+6); its product digit(a) digit(b) is
 *     congruent to a b mod m.  Two-digit moduli: d0 + 13 d1 as the two-limb
 *     family.
 *   - Products per output: ozemu_products_mixed(r) = min(r, 6) + 4 max(r-6, 0):
 *     r = 19 gives 58 products and, at k = 8192, the bit budget P = 88 that
 *     r = 13 three-limb moduli (117 products) give.
 *   - Limb planes: the single-digit moduli first, each [rows_p][k_p/2]
 *     (the digit of element k at row byte (k/128)*64 + (k%128)/2, two codes
 *     per byte, low nibble for even k); then the two-digit moduli, each
 *     [rows_p][k_p] in the two-limb layout.  Total: ozemu_plane_bytes_mixed.
 *   - Residue layout: as the three-limb calls, with these moduli (r of them).
 * Bit budget, rounding, CRT and scale-back are those of the other families
 * with these moduli.  Planes and residues of one family are not valid input
 * to another family's calls.  Arguments, ownership and errors are those of
 * the three-limb call of the same name, with r up to 20. */
int ozemu_max_moduli_mixed(void);          /* 20. host. */
int ozemu_single_digit_moduli_mixed(void); /* 6: moduli 0..5 are single-digit. host. */
int ozemu_moduli_mixed(int r, int32_t* out);
int ozemu_bit_budget_mixed(int k, int r, int* p_a, int* p_b);
size_t ozemu_plane_bytes_mixed(int rows, int k, int r);
/* FP4 products per output of the first r moduli; OZEMU_ERR_INVALID_ARG for r
 * out of range. host. */
int ozemu_products_mixed(int r);
int ozemu_split_rows_f64_mixed(int rows, int k, const double* X, int ldx, int p, int r,
                               uint8_t* planes, int32_t* shifts, cudaStream_t stream);
int ozemu_split_cols_f64_mixed(int k, int cols, const double* X, int ldx, int p, int r,
                               uint8_t* planes, int32_t* shifts, cudaStream_t stream);
/* Residues of C' = A'B' for the mixed-digit moduli: one launch of one FP4
 * product per K step for the single-digit moduli (exact FP32 accumulation
 * over chunks of 2^18, |digit| <= 8) and one of four products for the
 * two-digit ones. */
int ozemu_residue_gemm_mixed(int m, int n, int k, int r, const uint8_t* a_planes,
                             const uint8_t* b_planes, uint8_t* residues, cudaStream_t stream);
int ozemu_crt_f64_mixed(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a,
                        const int32_t* shifts_b, double* C, int ldc, cudaStream_t stream);

/* C = A B (device buffers, as ozemu_dgemm) through the mixed-digit stages.
 * Requires 2k < m_1...m_r of these moduli.  No narrow path; m >= 2048
 * pipelines the stages over row chunks like ozemu_dgemm.  Cached workspace. */
int ozemu_dgemm_mixed(int m, int n, int k, const double* A, int lda, const double* B,
                      int ldb, double* C, int ldc, int r, cudaStream_t stream);

/* ozemu_dgemm_mixed with HOST buffers, pipelined like ozemu_dgemm_host; the
 * result equals ozemu_dgemm_mixed's bit for bit. */
int ozemu_dgemm_host_mixed(int m, int n, int k, const double* A, int lda, const double* B,
                           int ldb, double* C, int ldc, int r, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* OZEMU_H */
