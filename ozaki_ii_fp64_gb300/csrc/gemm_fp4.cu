// FP4 limb GEMM on tcgen05: the 9 exact products of [AWE] abstract.
//
// A persistent grid (one CTA per SM) walks the (modulus l, 128 x BN output
// tile) pairs.  For every
// 128-wide K block the three A limb tiles and three B limb tiles (FP4 e2m1,
// K-major, 64-byte rows, 64-byte swizzle) arrive by TMA into a shared-memory
// stage; one thread issues the 9 limb products (2 MMAs of K = 64 each) into
// two TMEM accumulators, grouped by A limb so that the A-operand collector
// buffer serves the three products of each A tile from one shared-memory
// read, and folding the limb weights into the block scales:
//
//   D1 = A0B0 + 13 (A0B1 + A1B0)
//   D2 = A0B2 + A1B1 + A2B0 + 13 (A1B2 + A2B1) + 169 A2B2
//
// so sum_{i,j} 13^(i+j) A_i B_j = D1 + 169 D2.  Each digit d is stored as the
// FP4 value d/2; the UE4M3 scale 2 restores d and the scale 26 = 2 * 13
// applies the factor 13 (26 * 26 / 4 = 169).  Both scales and all products
// are exact, and the FP32 accumulators hold exact integers as long as they
// stay below 2^24: per K element |D1| grows by at most 64 + 2 * 13 * 64 =
// 1728 and |D2| by 80 + 2 * 13 * 8 + 169 = 457 for int8-range digits, so a
// chunk of 8192 K elements is exact.  Longer K is split into chunks: after
// each chunk the epilogue folds D1 + 169 D2 into a running value kept in a
// third TMEM region and the MMAs restart the accumulators.
//
// Two-limb moduli (m <= 113, residues in [-56, 56], digits |d0| <= 8,
// |d1| <= 4, no third limb): 4 products per K step.  The CTA-pair kernel
// folds all four into one accumulator, D = A0B0 + 13 (A0B1 + A1B0) +
// 169 A1B1 (A1's scale 26 in both of its products), which grows by at most
// 64 + 2 * 13 * 32 + 169 * 16 = 3600 per K element and so stays exact over
// chunks of 4096; with 224 columns per tile two accumulators fit in TMEM and
// alternate between tiles.  The single-CTA kernel keeps D1 and D2.
//
// The epilogue copies the accumulators to registers and releases them at
// once, so the next chunk's (or tile's) MMAs overlap the modular arithmetic
// and the stores; the TMA producer runs ahead across tiles through the
// shared-memory ring.
//
// The epilogue reduces D1 + 169 D2 modulo m_l ([AWE] abstract: the
// formulation holds modulo m) and stores a uint8 residue, or (INT8 product)
// forms the exact int32 sum.
//
// Warp roles (320 threads): warp 0 lane 0 = TMA producer; warp 1 = TMEM
// allocator, lane 0 = MMA issuer; warps 2..9 = epilogue (TMEM lane quarter
// = warp % 4, half of the tile's columns each).  Every wait is bounded in time; on expiry the kernel flags a
// time-out, drains what it issued, frees TMEM and exits.
#include <cstdint>
#include <cstdlib>
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kBM = 128;
constexpr int kBKBytes = 64;             // 128 FP4 elements per K block
constexpr int kATile = kBM * kBKBytes;   // 8 KB
constexpr int kEpiWarps = 8;             // two per TMEM lane quarter, each half of the columns
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kTmemCols = 512;
constexpr uint32_t kColD1 = 0, kColD2 = 128, kColRun = 256, kColSf2 = 384, kColSf26 = 416;
constexpr int kGroupM = 32;              // tile-row group for L2 reuse (32 x 1.5 MB of A planes stay resident)

template <int BN>
struct Cfg {
  static constexpr int kBTile = BN * kBKBytes;
  static constexpr int kStage = 3 * kATile + 3 * kBTile;
  static constexpr int kStages = (200 * 1024) / kStage > 8 ? 8 : (200 * 1024) / kStage;
  static constexpr int kSmem = 1024 + kStages * kStage + 256;
  static constexpr int kCols = BN / 2;   // accumulator columns per epilogue thread
};

struct GemmArgs {
  int m, n;
  int kb_total;    // 128-wide K blocks
  int kb_chunk;    // K blocks per exact chunk
  int rows_a_p, rows_b_p;
  int tiles_m, tiles_n;
  int total_tiles; // r * tiles_m * tiles_n
  EpiModuli em;
  uint8_t* res_out;
  long long ldr;
  int32_t* c32;
  long long ldc;
  uint32_t* flags;
};

// Lane 0 polls, the result is broadcast so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_word,
                                          uint32_t* flags) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_word, flags) ? 1 : 0;
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Bounded wait that ignores the abort word (used while draining).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint32_t* flags) {
  uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(flags, kFlagTimeout);
      return;
    }
  }
}

// x - m round(x / m) for an integer-valued |x| < 2^24: the quotient is
// rounded by adding 1.5 2^23 (one fma and one add on the full-rate pipes;
// a quotient off by one at a tie still leaves |result| <= m/2 + 1).
__device__ __forceinline__ float fmod_small(float x, float m, float inv_m) {
  const float q = fmaf(x, inv_m, 12582912.0f) - 12582912.0f;
  return fmaf(-q, m, x);
}

// The residue byte of an integer-valued v in [0, 256), without a conversion
// instruction: v + 2^23 holds v in its low mantissa bits.
__device__ __forceinline__ uint32_t byte_of_float(float v) { return __float_as_uint(v + 8388608.0f); }

// Tile t -> (modulus l, tile row tm, tile column tn): modulus-major, then
// groups of kGroupM tile rows swept column by column (L2 reuse).
__device__ __forceinline__ void tile_coords(int t, const GemmArgs& a, int& l, int& tm, int& tn) {
  const int per_mod = a.tiles_m * a.tiles_n;
  l = t / per_mod;
  const int u = t % per_mod;
  const int group = kGroupM * a.tiles_n;
  const int first_m = (u / group) * kGroupM;
  const int gm = min(kGroupM, a.tiles_m - first_m);
  tm = first_m + (u % group) % gm;
  tn = (u % group) / gm;
}

template <int CW>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&v)[CW]) {
#pragma unroll
  for (int c = 0; c < CW; c += 8) tmem_ld8(taddr + c, v + c);
}
template <int CW>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[CW]) {
#pragma unroll
  for (int c = 0; c < CW; c += 8) tmem_st8(taddr + c, v + c);
}

// NL: limbs per modulus (3; 2 for the two-limb moduli, whose third limb is 0:
// 4 products, the third limb neither loaded nor multiplied).
template <int BN, bool kResidue, int NL>
__global__ void __launch_bounds__(kThreads, 1)
    limb_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs args) {
  using C = Cfg<BN>;
  constexpr int CW = C::kCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* mma_done = tempty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // After a time-out anywhere on the device, later CTAs do no work (the flag
  // stays set until ozemu_get_status clears it).
  __shared__ int skip;
  if (threadIdx.x == 0) skip = (*reinterpret_cast<volatile uint32_t*>(args.flags) & kFlagTimeout) ? 1 : 0;
  __syncthreads();
  if (skip) return;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps);
    mbar_init(mma_done, 1);
    *abort_word = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  // Constant block scales: every byte of the two regions is 2.0 (0x40) or
  // 26.0 (0x5D) in UE4M3, so any scale-factor layout reads the same value.
  if (warp >= 2 && warp < 6) {
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0x40404040u;
    tmem_st16(tbase + lane_off + kColSf2, v);
    tmem_st16(tbase + lane_off + kColSf2 + 16, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0x5D5D5D5Du;
    tmem_st16(tbase + lane_off + kColSf26, v);
    tmem_st16(tbase + lane_off + kColSf26 + 16, v);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int kb_total = args.kb_total;
  const int n_chunks = (kb_total + args.kb_chunk - 1) / args.kb_chunk;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      int it = 0;  // K blocks issued by this CTA (across tiles)
      bool ok = true;
      for (int t = blockIdx.x; t < args.total_tiles && ok; t += gridDim.x) {
        int l, tm, tn;
        tile_coords(t, args, l, tm, tn);
        const int a_row = l * args.rows_a_p + tm * kBM;
        const int b_row = l * args.rows_b_p + tn * BN;
        for (int kb = 0; kb < kb_total; ++kb, ++it) {
          const int s = it % C::kStages;
          const uint32_t ph = (it / C::kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, abort_word, args.flags)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * C::kStage;
          mbar_arrive_expect_tx(&full[s], NL * (kATile + C::kBTile));
#pragma unroll
          for (int j = 0; j < NL; ++j)
            tma_load_2d(st + j * kATile, &tmA, &full[s], (NL * kb + j) * kBKBytes, a_row);
#pragma unroll
          for (int j = 0; j < NL; ++j)
            tma_load_2d(st + 3 * kATile + j * C::kBTile, &tmB, &full[s], (NL * kb + j) * kBKBytes, b_row);
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        for (int i = (it > C::kStages ? it - C::kStages : 0); i < it; ++i)
          drain_wait(&full[i % C::kStages], (i / C::kStages) & 1, args.flags);
      }
    }
    __syncwarp();  // the whole warp reaches the final barrier together
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_fp4(BN);
      const uint32_t d1 = tbase + kColD1, d2 = tbase + kColD2;
      const uint32_t s2 = tbase + kColSf2, s26 = tbase + kColSf26;
      int it = 0;  // K blocks consumed
      int g = 0;   // accumulator chunks produced
      bool ok = true;
      // Whether stage `it` is already known to be full: tested without
      // blocking while the previous stage's MMAs fill the (shallow) MMA
      // queue, so that a blocking wait, which lets the queue drain, is only
      // paid when the data is actually late.
      bool known_full = false;
      for (int t = blockIdx.x; t < args.total_tiles && ok; t += gridDim.x) {
        for (int c = 0; c < n_chunks && ok; ++c, ++g) {
          if (g > 0) {
            // The epilogue has copied the previous chunk out of TMEM.
            if (!mbar_wait(tempty, (g - 1) & 1, abort_word, args.flags)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const int kb0 = c * args.kb_chunk;
          const int kb1 = min(kb0 + args.kb_chunk, kb_total);
          for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % C::kStages;
            const uint32_t ph = (it / C::kStages) & 1;
            if (!known_full && !mbar_wait(&full[s], ph, abort_word, args.flags)) {
              ok = false;
              break;
            }
            known_full = false;
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * C::kStage);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const uint64_t a0 = smem_desc_sw64(st + 0 * kATile + ks * 32);
              const uint64_t a1 = smem_desc_sw64(st + 1 * kATile + ks * 32);
              const uint64_t a2 = smem_desc_sw64(st + 2 * kATile + ks * 32);
              const uint64_t b0 = smem_desc_sw64(st + 3 * kATile + 0 * C::kBTile + ks * 32);
              const uint64_t b1 = smem_desc_sw64(st + 3 * kATile + 1 * C::kBTile + ks * 32);
              const uint64_t b2 = smem_desc_sw64(st + 3 * kATile + 2 * C::kBTile + ks * 32);
              const uint32_t acc = (kb == kb0 && ks == 0) ? 0u : 1u;
              // Grouped by A limb so each A tile is read once per K step
              // (collector buffer), with one A scale per group: the factor
              // 13 sits on B's scale; A2 B2 (weight 169 = 26 * 26 / 4) needs
              // the other A scale and is issued on its own.
              if constexpr (NL == 3) {
                mma_fp4_fill(d1, a0, b0, idesc, s2, s2, acc);      // 1
                mma_fp4_use(d1, a0, b1, idesc, s2, s26, 1u);       // 13
                mma_fp4_lastuse(d2, a0, b2, idesc, s2, s2, acc);   // 1 (in D2)
                mma_fp4_fill(d1, a1, b0, idesc, s2, s26, 1u);      // 13
                mma_fp4_use(d2, a1, b1, idesc, s2, s2, 1u);        // 1 (in D2)
                mma_fp4_lastuse(d2, a1, b2, idesc, s2, s26, 1u);   // 13 (in D2)
                mma_fp4_fill(d2, a2, b0, idesc, s2, s2, 1u);       // 1 (in D2)
                mma_fp4_lastuse(d2, a2, b1, idesc, s2, s26, 1u);   // 13 (in D2)
                mma_fp4(d2, a2, b2, idesc, s26, s26, 1u);          // 169 (in D2)
              } else if constexpr (NL == 2) {
                // D1 = A0B0 + 13 (A0B1 + A1B0), D2 = A1B1 (weight 169 at the drain).
                mma_fp4_fill(d1, a0, b0, idesc, s2, s2, acc);      // 1
                mma_fp4_lastuse(d1, a0, b1, idesc, s2, s26, 1u);   // 13
                mma_fp4_fill(d1, a1, b0, idesc, s2, s26, 1u);      // 13
                mma_fp4_lastuse(d2, a1, b1, idesc, s2, s2, acc);   // 1 (in D2)
              } else {
                // Single-digit moduli: D1 = A0B0, the residue product itself.
                (void)a1; (void)a2; (void)b1; (void)b2;
                mma_fp4(d1, a0, b0, idesc, s2, s2, acc);           // 1
              }
              if (ks == 0)
                known_full = mbar_test_wait(&full[(it + 1) % C::kStages], ((it + 1) / C::kStages) & 1);
            }
            tc_commit(&empty[s]);
          }
          if (ok) tc_commit(tfull);
        }
      }
      // All MMAs issued by this thread complete before teardown.
      tc_commit(mma_done);
      drain_wait(mma_done, 0, args.flags);
    }
    __syncwarp();  // the whole warp reaches the final barrier together
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(half * CW);
    int g = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < args.total_tiles && ok; t += gridDim.x) {
      int l, tm, tn;
      tile_coords(t, args, l, tm, tn);
      const int grow = tm * kBM + quarter * 32 + lane;
      const float fm = args.em.m[l], finv = args.em.inv_m[l], fw = args.em.w169[l];
      for (int c = 0; c < n_chunks; ++c, ++g) {
        if (!warp_wait(tfull, g & 1, abort_word, args.flags)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v1[CW], v2[CW];
        tmem_ld_cols<CW>(tbase + lane_off + kColD1 + col0, v1);
        if constexpr (NL == 1) {
#pragma unroll
          for (int i = 0; i < CW; ++i) v2[i] = 0u;  // single-digit moduli: no D2 (0.0f)
        } else {
          tmem_ld_cols<CW>(tbase + lane_off + kColD2 + col0, v2);
        }
        tmem_wait_ld();
        // Accumulators copied: the next chunk's MMAs may start.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty);

        const bool last = (c == n_chunks - 1);
        uint32_t out[CW];
        if constexpr (kResidue) {
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            const float r1 = fmod_small(__uint_as_float(v1[i]), fm, finv);
            const float r2 = fmod_small(__uint_as_float(v2[i]), fm, finv);
            out[i] = __float_as_uint(fmaf(r2, fw, r1));  // |.| < 2^17, exact
          }
        } else {
#pragma unroll
          for (int i = 0; i < CW; ++i)
            out[i] = static_cast<uint32_t>(__float2int_rn(__uint_as_float(v1[i])) +
                                           169 * __float2int_rn(__uint_as_float(v2[i])));
        }
        if (c > 0) {
          tmem_ld_cols<CW>(tbase + lane_off + kColRun + col0, v1);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            if constexpr (kResidue)
              out[i] = __float_as_uint(__uint_as_float(out[i]) + __uint_as_float(v1[i]));
            else
              out[i] = static_cast<uint32_t>(static_cast<int>(out[i]) + static_cast<int>(v1[i]));
          }
        }
        if constexpr (kResidue) {
#pragma unroll
          for (int i = 0; i < CW; ++i) {
            float v = fmod_small(__uint_as_float(out[i]), fm, finv);
            v = v < 0.f ? v + fm : v;  // [0, m)
            out[i] = last ? static_cast<uint32_t>(__float2int_rn(v)) : __float_as_uint(v);
          }
        }
        if (!last) {
          tmem_st_cols<CW>(tbase + lane_off + kColRun + col0, out);
          tmem_wait_st();
          continue;
        }
        if (grow >= args.m) continue;
        const int gcol0 = tn * BN + static_cast<int>(col0);
        if constexpr (kResidue) {
          uint8_t* rrow = args.res_out + (static_cast<long long>(l) * args.m + grow) * args.ldr;
#pragma unroll
          for (int q = 0; q < CW; q += 16) {
            if (CW >= 16) {
              if (gcol0 + q < args.ldr) {
                uint4 w;
                w.x = out[q + 0] | (out[q + 1] << 8) | (out[q + 2] << 16) | (out[q + 3] << 24);
                w.y = out[q + 4] | (out[q + 5] << 8) | (out[q + 6] << 16) | (out[q + 7] << 24);
                w.z = out[q + 8] | (out[q + 9] << 8) | (out[q + 10] << 16) | (out[q + 11] << 24);
                w.w = out[q + 12] | (out[q + 13] << 8) | (out[q + 14] << 16) | (out[q + 15] << 24);
                *reinterpret_cast<uint4*>(rrow + gcol0 + q) = w;
              }
            } else {
              if (gcol0 < args.ldr) {
                uint2 w;
                w.x = out[0] | (out[1] << 8) | (out[2] << 16) | (out[3] << 24);
                w.y = out[4] | (out[5] << 8) | (out[6] << 16) | (out[7] << 24);
                *reinterpret_cast<uint2*>(rrow + gcol0) = w;
              }
            }
          }
        } else {
          int32_t* crow = args.c32 + static_cast<long long>(grow) * args.ldc;
          const bool vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.c32) & 15u) == 0);
#pragma unroll
          for (int q = 0; q < CW; q += 4) {
            const int col = gcol0 + q;
            if (vec && col + 4 <= args.n) {
              *reinterpret_cast<int4*>(crow + col) =
                  make_int4(static_cast<int>(out[q]), static_cast<int>(out[q + 1]), static_cast<int>(out[q + 2]),
                            static_cast<int>(out[q + 3]));
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (col + i < args.n) crow[col + i] = static_cast<int32_t>(out[q + i]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair variant: the two CTAs of a cluster compute one 256 x 224 tile with
// the 2-SM form of the MMA (M = 256): each CTA holds its 128 rows of the A
// limb tiles and one half (112 rows) of the B limb tiles.  Each MMA then does
// 1.75x the work of a 128 x 128 one per A-tile read and per stage barrier:
// the 128 x 128 single-CTA MMA reads shared memory at about the full port
// rate, which leaves no room for the TMA fills and barrier reads.
// Used for residue products with n > 64; for K beyond one exact chunk each
// chunk is an accumulation round whose residues the epilogue adds, modulo
// m_l, to the ones it keeps in registers (four per register).
// ---------------------------------------------------------------------------
constexpr int kBN2 = kPairTileCols;              // pair tile N (224)
constexpr int kBHalf = kBN2 / 2;                 // B rows per CTA
constexpr int kBTile2 = kBHalf * kBKBytes;       // 7168 B
// A stage holds kKpS 128-wide K blocks: the NL A limb tiles of each, then
// the NL B limb tiles of each; the ring keeps 180 KB of them in flight for
// every NL (4 stages of three limbs, 6 of two, 3 of four single-digit K
// blocks).  Single-digit moduli take 4 K blocks per stage so that each stage
// barrier serves 8 MMAs, as a two-limb stage does: with one K block (2 MMAs)
// per barrier the issuing thread's wait and commit per stage left the tensor
// pipe idle most of the time.
template <int NL>
struct PairCfg {
  static constexpr int kKpS = NL == 1 ? 4 : 1;  // K blocks per stage
  static constexpr int kStage = kKpS * NL * (kATile + kBTile2);
  static constexpr int kStages = (180 * 1024) / kStage;
  static constexpr int kSmem = 1024 + kStages * kStage + 256;
};
constexpr int kSmem2 = PairCfg<3>::kSmem;
static_assert(PairCfg<1>::kSmem == kSmem2 && PairCfg<2>::kSmem == kSmem2, "one shared-memory size for every NL");
constexpr int kTmemCols2 = 512;
constexpr uint32_t kColD1p = 0, kColD2p = 224, kColSf2p = 448, kColSf26p = 464;
// INT4 x INT8 (four planes, NL = 4): the slot at kColSf26p holds 12 instead
// of 26, and two more slots hold 4 and 6, so that each plane product k gets
// scales whose product is 4 g_k (FP4 holds half the digit): (2, 6), (2, 4),
// (4, 6), (4, 12) for g = (3, 2, 6, 12).
constexpr uint32_t kColSf4p = 480, kColSf6p = 496;
constexpr int kPairCols = kBN2 / 2;              // accumulator columns per epilogue thread (two per lane quarter)
constexpr int kGroupM2 = 16;                     // pair-tile rows per raster group

struct PairArgs {
  int m, n, kb_total;
  int kc_blocks;  // 128-wide K blocks per exactly accumulated chunk
  int rows_a_p, rows_b_p;
  int tiles_m2, tiles_n2, total_tiles;
  EpiModuli em;
  uint8_t* res_out;
  long long ldr;
  int32_t* c32;   // INT8 mode: C32 = D1 + 169 D2, leading dimension ldc
  long long ldc;
  uint32_t* flags;
};

__device__ __forceinline__ void pair_tile_coords(int t, const PairArgs& a, int& l, int& tm2, int& tn) {
  const int per_mod = a.tiles_m2 * a.tiles_n2;
  l = t / per_mod;
  const int u = t % per_mod;
  const int group = kGroupM2 * a.tiles_n2;
  const int first_m = (u / group) * kGroupM2;
  const int gm = min(kGroupM2, a.tiles_m2 - first_m);
  tm2 = first_m + (u % group) % gm;
  tn = (u % group) / gm;
}

// After an abort, give copies already issued (whose completion may be
// signalled in the other CTA) time to land before the pair tears down.
__device__ __forceinline__ void settle_after_abort() {
  const uint64_t t0 = globaltimer();
  while (globaltimer() - t0 < 50000ull) {
  }
}

// kInt: the INT8 product (r = 1, one exact K chunk): the epilogue writes the
// int32 sums D1 + 169 D2 slice by slice instead of residues.
template <bool kInt, int NL>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    limb_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const PairArgs args) {
  constexpr int kStage2 = PairCfg<NL>::kStage;
  constexpr int kStages2 = PairCfg<NL>::kStages;
  constexpr int kKpS = PairCfg<NL>::kKpS;
  constexpr int kATiles = kKpS * NL;  // A tiles per stage (B tiles follow them)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages2 * kStage2);
  uint64_t* empty = full + kStages2;
  // Accumulator hand-off, per TMEM buffer (two-limb moduli: two buffers).
  uint64_t* tfull = empty + kStages2;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile int* abort_word = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = (rank == 0);
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  // Three-limb moduli: D1 and D2 fill 448 of the 512 TMEM columns, one tile
  // at a time.  Two-limb moduli: one accumulator D = D1 + 169 D2 per tile
  // (exact for K chunks of 4096); single-digit moduli: one accumulator
  // D = A0 B0.  Then two tiles' accumulators alternate and the MMAs of one
  // round run while the epilogue drains the other.
  constexpr int kBufs = (NL <= 2 || NL == 4) ? 2 : 1;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kStages2; ++s) {
      mbar_init(&full[s], 1);   // armed by the first CTA with both CTAs' bytes
      mbar_init(&empty[s], 1);  // one commit from the pair's MMA issuer
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * kEpiWarps);
    }
    mbar_init(mma_done, 1);
    *abort_word = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kTmemCols2);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  if (warp >= 2 && warp < 6) {
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint32_t v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0x40404040u;
    tmem_st16(tbase + lane_off + kColSf2p, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = NL == 4 ? 0x54545454u : 0x5D5D5D5Du;  // 12 or 26
    tmem_st16(tbase + lane_off + kColSf26p, v);
    if constexpr (NL == 4) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0x48484848u;  // 4
      tmem_st16(tbase + lane_off + kColSf4p, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0x4C4C4C4Cu;  // 6
      tmem_st16(tbase + lane_off + kColSf6p, v);
    }
    tmem_wait_st();
  }
  // Both CTAs' barriers initialised and scales written before any remote
  // signal or pair MMA.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();

  const int kb_total = args.kb_total;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      int it = 0;
      bool ok = true;
      for (int t = pair; t < args.total_tiles && ok; t += npairs) {
        int l, tm2, tn;
        pair_tile_coords(t, args, l, tm2, tn);
        const int a_row = l * args.rows_a_p + tm2 * 256 + static_cast<int>(rank) * kBM;
        const int b_row = l * args.rows_b_p + tn * kBN2 + static_cast<int>(rank) * kBHalf;
        for (int kc0 = 0; kc0 < kb_total && ok; kc0 += args.kc_blocks) {
          const int kc1 = kc0 + args.kc_blocks < kb_total ? kc0 + args.kc_blocks : kb_total;
          for (int kb = kc0; kb < kc1; kb += kKpS, ++it) {
            const int nb = kc1 - kb < kKpS ? kc1 - kb : kKpS;  // K blocks in this stage
            const int s = it % kStages2;
            const uint32_t ph = (it / kStages2) & 1;
            if (!mbar_wait(&empty[s], ph ^ 1, abort_word, args.flags)) {
              ok = false;
              break;
            }
            uint8_t* st = smem + s * kStage2;
            const uint32_t full_leader = mapa_shared(&full[s], 0);
            // Only the first CTA arms the barrier (with both CTAs' bytes): a
            // remote release-arrive from the second CTA would wait for its
            // earlier bulk copies and serialise the stages.  The phase cannot
            // complete before it is armed, and the second CTA cannot fill a
            // stage of the next phase before the pair's MMAs freed it.
            if (leader) mbar_arrive_expect_tx(&full[s], 2 * nb * NL * (kATile + kBTile2));
            for (int q = 0; q < nb; ++q) {
#pragma unroll
              for (int j = 0; j < NL; ++j)
                tma_load_2d_pair(st + (q * NL + j) * kATile, &tmA, full_leader, (NL * (kb + q) + j) * kBKBytes,
                                 a_row);
#pragma unroll
              for (int j = 0; j < NL; ++j)
                tma_load_2d_pair(st + kATiles * kATile + (q * NL + j) * kBTile2, &tmB, full_leader,
                                 (NL * (kb + q) + j) * kBKBytes, b_row);
            }
          }
        }
      }
      if (!ok) settle_after_abort();
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_fp4(kBN2, 256);
      const uint32_t d1 = tbase + kColD1p, d2 = tbase + kColD2p;
      const uint32_t s2 = tbase + kColSf2p, s26 = tbase + kColSf26p;
      int it = 0, g = 0;
      bool ok = true;
      bool known_full = false;
      // g counts accumulation rounds: one per K chunk of each tile.
      for (int t = pair; t < args.total_tiles && ok; t += npairs) {
        for (int kc0 = 0; kc0 < kb_total && ok; kc0 += args.kc_blocks, ++g) {
          // Round g fills buffer g % kBufs for its (g / kBufs)-th time; the
          // epilogue must have released that buffer's previous round.
          const int buf = g % kBufs, use = g / kBufs;
          if (use > 0) {
            if (!mbar_wait(&tempty[buf], (use - 1) & 1, abort_word, args.flags)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t dacc = tbase + static_cast<uint32_t>(buf * kBN2);  // two-limb accumulator
          const int kc1 = kc0 + args.kc_blocks < kb_total ? kc0 + args.kc_blocks : kb_total;
          for (int kb = kc0; kb < kc1; kb += kKpS, ++it) {
            const int s = it % kStages2;
            const uint32_t ph = (it / kStages2) & 1;
            if (!known_full && !mbar_wait(&full[s], ph, abort_word, args.flags)) {
              ok = false;
              break;
            }
            known_full = false;
            tc_fence_after();
            const uint32_t st = smem_u32(smem + s * kStage2);
            if constexpr (NL == 4) {
              // INT4 x INT8: D = sum_k g_k A_k B_k over the four planes, the
              // weights carried by the scale pairs.
              const uint32_t s4 = tbase + kColSf4p, s6 = tbase + kColSf6p, s12 = tbase + kColSf26p;
#pragma unroll
              for (int ks = 0; ks < 2; ++ks) {
                uint64_t a[4], b[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  a[j] = smem_desc_sw64(st + j * kATile + ks * 32);
                  b[j] = smem_desc_sw64(st + 4 * kATile + j * kBTile2 + ks * 32);
                }
                const uint32_t acc = (kb == kc0 && ks == 0) ? 0u : 1u;
                mma_fp4_pair(dacc, a[0], b[0], idesc, s2, s6, acc);  // 3
                mma_fp4_pair(dacc, a[1], b[1], idesc, s2, s4, 1u);   // 2
                mma_fp4_pair(dacc, a[2], b[2], idesc, s4, s6, 1u);   // 6
                mma_fp4_pair(dacc, a[3], b[3], idesc, s4, s12, 1u);  // 12
                if (ks == 0)
                  known_full = mbar_test_wait(&full[(it + 1) % kStages2], ((it + 1) / kStages2) & 1);
              }
              tc_commit_pair_multicast(&empty[s], 0x3);
              continue;
            }
            if constexpr (NL == 1) {
              // Single-digit moduli: D = A0 B0, the residue product itself,
              // over the stage's nb K blocks.
              const int nb = kc1 - kb < kKpS ? kc1 - kb : kKpS;
              for (int q = 0; q < nb; ++q) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                  const uint64_t a0 = smem_desc_sw64(st + q * kATile + ks * 32);
                  const uint64_t b0 = smem_desc_sw64(st + kATiles * kATile + q * kBTile2 + ks * 32);
                  const uint32_t acc = (kb == kc0 && q == 0 && ks == 0) ? 0u : 1u;
                  mma_fp4_pair(dacc, a0, b0, idesc, s2, s2, acc);  // 1
                }
              }
              known_full = mbar_test_wait(&full[(it + 1) % kStages2], ((it + 1) / kStages2) & 1);
              tc_commit_pair_multicast(&empty[s], 0x3);
              continue;
            }
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
              const uint64_t a0 = smem_desc_sw64(st + 0 * kATile + ks * 32);
              const uint64_t a1 = smem_desc_sw64(st + 1 * kATile + ks * 32);
              const uint64_t a2 = smem_desc_sw64(st + 2 * kATile + ks * 32);
              const uint64_t b0 = smem_desc_sw64(st + NL * kATile + 0 * kBTile2 + ks * 32);
              const uint64_t b1 = smem_desc_sw64(st + NL * kATile + 1 * kBTile2 + ks * 32);
              const uint64_t b2 = smem_desc_sw64(st + NL * kATile + 2 * kBTile2 + ks * 32);
              const uint32_t acc = (kb == kc0 && ks == 0) ? 0u : 1u;
              if constexpr (NL == 3) {
                mma_fp4_pair_fill(d1, a0, b0, idesc, s2, s2, acc);      // 1
                mma_fp4_pair_use(d1, a0, b1, idesc, s2, s26, 1u);       // 13
                mma_fp4_pair_lastuse(d2, a0, b2, idesc, s2, s2, acc);   // 1 (in D2)
                mma_fp4_pair_fill(d1, a1, b0, idesc, s2, s26, 1u);      // 13
                mma_fp4_pair_use(d2, a1, b1, idesc, s2, s2, 1u);        // 1 (in D2)
                mma_fp4_pair_lastuse(d2, a1, b2, idesc, s2, s26, 1u);   // 13 (in D2)
                mma_fp4_pair_fill(d2, a2, b0, idesc, s2, s2, 1u);       // 1 (in D2)
                mma_fp4_pair_lastuse(d2, a2, b1, idesc, s2, s26, 1u);   // 13 (in D2)
                mma_fp4_pair(d2, a2, b2, idesc, s26, s26, 1u);          // 169 (in D2)
              } else {
                // One accumulator D = A0B0 + 13 (A0B1 + A1B0) + 169 A1B1: A1
                // carries the scale 26 in both of its products.
                mma_fp4_pair_fill(dacc, a0, b0, idesc, s2, s2, acc);       // 1
                mma_fp4_pair_lastuse(dacc, a0, b1, idesc, s2, s26, 1u);    // 13
                mma_fp4_pair_fill(dacc, a1, b0, idesc, s26, s2, 1u);       // 13
                mma_fp4_pair_lastuse(dacc, a1, b1, idesc, s26, s26, 1u);   // 169
              }
              if (ks == 0)
                known_full = mbar_test_wait(&full[(it + 1) % kStages2], ((it + 1) / kStages2) & 1);
            }
            tc_commit_pair_multicast(&empty[s], 0x3);
          }
          if (ok) tc_commit_pair_multicast(&tfull[buf], 0x3);
        }
      }
      tc_commit_pair_multicast(mma_done, 0x1);
      drain_wait(mma_done, 0, args.flags);
      if (!ok) settle_after_abort();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // 112 columns per thread: fold D1, D2 to residues 16 columns at a time
    // (packed four to a register), release TMEM, then store.
    constexpr int CW = kPairCols;
    constexpr int kSlice = 16;
    const int ew = warp - 2;
    const int quarter = warp & 3;
    const int half = ew >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t col0 = static_cast<uint32_t>(half * CW);
    int g = 0;  // accumulation rounds, as counted by the MMA issuer
    bool live = true;
    for (int t = pair; t < args.total_tiles && live; t += npairs) {
      int l, tm2, tn;
      pair_tile_coords(t, args, l, tm2, tn);
      const int grow = tm2 * 256 + static_cast<int>(rank) * kBM + quarter * 32 + lane;
      const float fm = args.em.m[l], finv = args.em.inv_m[l], fw = args.em.w169[l];
      // Residues of this thread's 112 outputs, four to a register; chunks
      // after the first are added to them modulo m.
      uint32_t packed[CW / 4];
      for (int kc0 = 0; kc0 < kb_total; kc0 += args.kc_blocks, ++g) {
        const bool first = (kc0 == 0);
        const int buf = g % kBufs, use = g / kBufs;
        if (!warp_wait(&tfull[buf], use & 1, abort_word, args.flags)) {
          live = false;
          break;
        }
        tc_fence_after();
        if constexpr (NL == 4) {
          // INT4 x INT8: one accumulator, exact below 2^24 for K chunks of
          // 8192 (|a b| <= 1024); the int32 sums of the chunks add up in C32.
          const uint32_t dcol = tbase + lane_off + static_cast<uint32_t>(buf * kBN2) + col0;
          uint32_t v1[kSlice], n1[kSlice];
          tmem_ld_cols<kSlice>(dcol, n1);
#pragma unroll
          for (int c = 0; c < CW; c += kSlice) {
            tmem_wait_ld_regs(n1);
#pragma unroll
            for (int i = 0; i < kSlice; ++i) v1[i] = n1[i];
            if (c + kSlice < CW) tmem_ld_cols<kSlice>(dcol + c + kSlice, n1);
            if (grow < args.m) {
              int32_t* crow = args.c32 + static_cast<long long>(grow) * args.ldc;
              const int col = tn * kBN2 + static_cast<int>(col0) + c;
#pragma unroll
              for (int i = 0; i < kSlice; ++i) {
                if (col + i < args.n) {
                  const int v = __float2int_rn(__uint_as_float(v1[i]));
                  crow[col + i] = first ? v : crow[col + i] + v;
                }
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(&tempty[buf], 0));
          continue;
        }
        if constexpr (NL <= 2) {
          // One accumulator (|D| < 3600 * 4096 < 2^24 for two-limb moduli,
          // 64 * 2^18 for single-digit ones): one reduction modulo m.
          const uint32_t dcol = tbase + lane_off + static_cast<uint32_t>(buf * kBN2) + col0;
          uint32_t v1[kSlice], n1[kSlice];
          tmem_ld_cols<kSlice>(dcol, n1);
#pragma unroll
          for (int c = 0; c < CW; c += kSlice) {
            tmem_wait_ld_regs(n1);
#pragma unroll
            for (int i = 0; i < kSlice; ++i) v1[i] = n1[i];
            if (c + kSlice < CW) tmem_ld_cols<kSlice>(dcol + c + kSlice, n1);
#pragma unroll
            for (int i = 0; i < kSlice; i += 4) {
              uint32_t b[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float v = fmod_small(__uint_as_float(v1[i + e]), fm, finv);
                v = v < 0.f ? v + fm : v;
                if (!first) {
                  v += __uint_as_float(__byte_perm(packed[(c + i) / 4], 0x4B000000u, 0x7650u | (e & 3))) - 8388608.0f;
                  v = v >= fm ? v - fm : v;
                }
                b[e] = byte_of_float(v);
              }
              packed[(c + i) / 4] =
                  __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(&tempty[buf], 0));
          continue;
        }
        // Slice c + 1 is loaded from TMEM while slice c is folded.
        uint32_t v1[kSlice], v2[kSlice], n1[kSlice], n2[kSlice];
        tmem_ld_cols<kSlice>(tbase + lane_off + kColD1p + col0, n1);
        tmem_ld_cols<kSlice>(tbase + lane_off + kColD2p + col0, n2);
#pragma unroll
        for (int c = 0; c < CW; c += kSlice) {
          tmem_wait_ld_regs(n1, n2);
#pragma unroll
          for (int i = 0; i < kSlice; ++i) {
            v1[i] = n1[i];
            v2[i] = n2[i];
          }
          if (c + kSlice < CW) {
            tmem_ld_cols<kSlice>(tbase + lane_off + kColD1p + col0 + c + kSlice, n1);
            tmem_ld_cols<kSlice>(tbase + lane_off + kColD2p + col0 + c + kSlice, n2);
          }
          if constexpr (kInt) {
            if (grow < args.m) {
              int32_t* crow = args.c32 + static_cast<long long>(grow) * args.ldc;
              const int col = tn * kBN2 + static_cast<int>(col0) + c;
              int v[kSlice];
#pragma unroll
              for (int i = 0; i < kSlice; ++i)
                v[i] = __float2int_rn(__uint_as_float(v1[i])) + 169 * __float2int_rn(__uint_as_float(v2[i]));
              if (((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.c32) & 15u) == 0) &&
                  col + kSlice <= args.n) {
#pragma unroll
                for (int q = 0; q < kSlice; q += 4)
                  *reinterpret_cast<int4*>(crow + col + q) = make_int4(v[q], v[q + 1], v[q + 2], v[q + 3]);
              } else {
#pragma unroll
                for (int i = 0; i < kSlice; ++i)
                  if (col + i < args.n) crow[col + i] = v[i];
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < kSlice; i += 4) {
              uint32_t b[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // |D1| <= 1728 * 8192 and |r2 w169| <= 129 * 128, so D1 + r2 w169 stays
                // below 2^24 and exact.
                const float r2 = fmod_small(__uint_as_float(v2[i + e]), fm, finv);
                float v = fmod_small(fmaf(r2, fw, __uint_as_float(v1[i + e])), fm, finv);
                v = v < 0.f ? v + fm : v;
                if (!first) {  // + the residue of the earlier chunks, modulo m
                  v += __uint_as_float(__byte_perm(packed[(c + i) / 4], 0x4B000000u, 0x7650u | (e & 3))) - 8388608.0f;
                  v = v >= fm ? v - fm : v;
                }
                b[e] = byte_of_float(v);
              }
              packed[(c + i) / 4] =
                  __byte_perm(__byte_perm(b[0], b[1], 0x0040), __byte_perm(b[2], b[3], 0x0040), 0x5410);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(&tempty[buf], 0));
      }
      if (kInt || !live || grow >= args.m) continue;
      uint8_t* rrow = args.res_out + (static_cast<long long>(l) * args.m + grow) * args.ldr;
      const int gcol0 = tn * kBN2 + static_cast<int>(col0);
#pragma unroll
      for (int q = 0; q < CW; q += 16) {
        if (gcol0 + q < args.ldr)
          *reinterpret_cast<uint4*>(rrow + gcol0 + q) =
              make_uint4(packed[q / 4], packed[q / 4 + 1], packed[q / 4 + 2], packed[q / 4 + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the pair's MMAs, commits and remote signals are all done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, kTmemCols2);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D map over the limb planes of r moduli: y = modulus l rows_p + row;
// x = byte within the row, where the three limbs of 128-element K block kb
// lie at x = (3 kb + j) 64 (two-limb moduli: (2 kb + j) 64).
bool make_plane_map(CUtensorMap* map, const uint8_t* base, int k_p, int limbs, long long total_rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const long long row_bytes = static_cast<long long>(limbs) * k_p / 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(total_rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, bool kResidue, int NL>
cudaError_t launch_bn(const LimbGemmCall& c, cudaStream_t stream) {
  using Cf = Cfg<BN>;
  const int rows_a_p = round_up(c.m, kRowAlign), rows_b_p = round_up(c.n, kRowAlign);
  const int k_p = round_up(c.k, kKAlign);
  const int r = c.residue_mode ? c.r : 1;
  CUtensorMap ma, mb;
  if (!make_plane_map(&ma, c.a_planes, k_p, NL, 1LL * r * rows_a_p, kBM)) return cudaErrorInvalidValue;
  if (!make_plane_map(&mb, c.b_planes, k_p, NL, 1LL * r * rows_b_p, BN)) return cudaErrorInvalidValue;
  GemmArgs a;
  a.m = c.m;
  a.n = c.n;
  a.kb_total = k_p / 128;
  a.kb_chunk = c.kc_blocks;
  a.rows_a_p = rows_a_p;
  a.rows_b_p = rows_b_p;
  a.tiles_m = (c.m + kBM - 1) / kBM;
  a.tiles_n = (c.n + BN - 1) / BN;
  a.total_tiles = r * a.tiles_m * a.tiles_n;
  a.em = c.em;
  a.res_out = c.res_out;
  a.ldr = c.ldr;
  a.c32 = c.c32;
  a.ldc = c.ldc;
  a.flags = c.flags;
  auto kern = limb_gemm_kernel<BN, kResidue, NL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.total_tiles < sms ? a.total_tiles : sms;  // persistent: one CTA per SM
  kern<<<grid, kThreads, Cf::kSmem, stream>>>(ma, mb, a);
  return cudaGetLastError();
}

template <bool kInt, int NL>
cudaError_t launch_pair(const LimbGemmCall& c, cudaStream_t stream) {
  const int rows_a_p = round_up(c.m, kRowAlign), rows_b_p = round_up(c.n, kRowAlign);
  const int k_p = round_up(c.k, kKAlign);
  CUtensorMap ma, mb;
  if (!make_plane_map(&ma, c.a_planes, k_p, NL, 1LL * c.r * rows_a_p, kBM)) return cudaErrorInvalidValue;
  if (!make_plane_map(&mb, c.b_planes, k_p, NL, 1LL * c.r * rows_b_p, kBHalf)) return cudaErrorInvalidValue;
  PairArgs a;
  a.m = c.m;
  a.n = c.n;
  a.kb_total = k_p / 128;
  // Two-limb moduli: one accumulator, exact for chunks of 4096 (32 blocks).
  // Single-digit moduli (|digit| <= 8): |D| grows by at most 64 per K
  // element, so chunks of 2^18 (2048 blocks) are exact.
  a.kc_blocks = (NL == 2 && c.kc_blocks > 32) ? 32 : c.kc_blocks;
  if (NL == 1) a.kc_blocks = a.kb_total < 2048 ? a.kb_total : 2048;
  if (NL == 4 && a.kc_blocks > 64) a.kc_blocks = 64;
  a.rows_a_p = rows_a_p;
  a.rows_b_p = rows_b_p;
  a.tiles_m2 = (c.m + 255) / 256;
  a.tiles_n2 = (c.n + kBN2 - 1) / kBN2;
  a.total_tiles = c.r * a.tiles_m2 * a.tiles_n2;
  a.em = c.em;
  a.res_out = c.res_out;
  a.ldr = c.ldr;
  a.c32 = c.c32;
  a.ldc = c.ldc;
  a.flags = c.flags;
  cudaError_t e =
      cudaFuncSetAttribute(limb_gemm_pair_kernel<kInt, NL>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem2);
  if (e != cudaSuccess) return e;
  // A persistent grid must not exceed the clusters that can be resident at
  // once, or the excess clusters start only when others finish.
  static int max_pairs[64] = {0};  // every instantiation has the same resources
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (max_pairs[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmem2;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, limb_gemm_pair_kernel<kInt, NL>, &cfg);
    if (e != cudaSuccess || n < 1) {
      cudaGetLastError();
      int sms = 148;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      n = sms / 2;
    }
    max_pairs[dev] = n;
  }
  const int pairs = a.total_tiles < max_pairs[dev] ? a.total_tiles : max_pairs[dev];
  limb_gemm_pair_kernel<kInt, NL><<<2 * pairs, kThreads, kSmem2, stream>>>(ma, mb, a);
  return cudaGetLastError();
}

bool use_pair(const LimbGemmCall& c) {
  if (c.n <= 64 || c.kc_blocks < 1) return false;
  // The INT8 product keeps no running value across K chunks in this kernel.
  if (!c.residue_mode && round_up(c.k, kKAlign) / 128 > c.kc_blocks) return false;
  if (const char* s = std::getenv("OZEMU_GEMM_PAIR")) return s[0] != '0';
  return true;
}

template <bool kResidue, int NL>
cudaError_t launch_mode(const LimbGemmCall& c, cudaStream_t stream) {
  if (c.n <= 16) return launch_bn<16, kResidue, NL>(c, stream);
  if (c.n <= 32) return launch_bn<32, kResidue, NL>(c, stream);
  if (c.n <= 64) return launch_bn<64, kResidue, NL>(c, stream);
  return launch_bn<128, kResidue, NL>(c, stream);
}

}  // namespace

cudaError_t launch_limb_gemm(const LimbGemmCall& call, cudaStream_t stream) {
  if (call.limbs == 2) {  // two-limb moduli: residue products only
    if (!call.residue_mode) return cudaErrorInvalidValue;
    return use_pair(call) ? launch_pair<false, 2>(call, stream) : launch_mode<true, 2>(call, stream);
  }
  if (call.limbs == 4) {  // INT4 x INT8 planes: int32 products only, any n
    if (call.residue_mode || call.kc_blocks < 1) return cudaErrorInvalidValue;
    return launch_pair<true, 4>(call, stream);
  }
  if (call.limbs == 1) {  // single-digit moduli: residue products only
    if (!call.residue_mode) return cudaErrorInvalidValue;
    return use_pair(call) ? launch_pair<false, 1>(call, stream) : launch_mode<true, 1>(call, stream);
  }
  if (call.limbs != 3) return cudaErrorInvalidValue;
  if (use_pair(call))
    return call.residue_mode ? launch_pair<false, 3>(call, stream) : launch_pair<true, 3>(call, stream);
  return call.residue_mode ? launch_mode<true, 3>(call, stream) : launch_mode<false, 3>(call, stream);
}

}  // namespace ozemu
