// FP4 limb GEMM on tcgen05: the 9 exact products of [AWE] abstract.
//
// One CTA computes one 128 x BN output tile for one modulus l.  For every
// 128-wide K block the three A limb tiles and three B limb tiles (FP4 e2m1,
// K-major, 64-byte rows, 64-byte swizzle) arrive by TMA into a shared-memory
// stage; one thread issues the 9 limb products (2 MMAs of K = 64 each) into
// two TMEM accumulators, folding the limb weights into the block scales:
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
// The epilogue reduces D1 + 169 D2 modulo m_l ([AWE] abstract: the
// formulation holds modulo m) and stores a uint8 residue, or (INT8 product)
// forms the exact int32 sum.
//
// Warp roles (192 threads): warp 0 lane 0 = TMA producer; warp 1 = TMEM
// allocator, lane 0 = MMA issuer; warps 2..5 = epilogue (TMEM lane quarter
// = warp % 4).  Every wait is bounded in time; on expiry the kernel flags a
// time-out, drains what it issued, frees TMEM and exits.
#include <cstdint>
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace ozemu {

namespace {

constexpr int kBM = 128;
constexpr int kBKBytes = 64;             // 128 FP4 elements per K block
constexpr int kATile = kBM * kBKBytes;   // 8 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr uint32_t kColD1 = 0, kColD2 = 128, kColRun = 256, kColSf2 = 384, kColSf26 = 416;
constexpr int kGroupM = 8;               // tile-row group for L2 reuse

template <int BN>
struct Cfg {
  static constexpr int kBTile = BN * kBKBytes;
  static constexpr int kStage = 3 * kATile + 3 * kBTile;
  static constexpr int kStages = (200 * 1024) / kStage > 8 ? 8 : (200 * 1024) / kStage;
  static constexpr int kSmem = 1024 + kStages * kStage + 256;
};

struct GemmArgs {
  int m, n;
  int kb_total;    // 128-wide K blocks
  int kb_chunk;    // K blocks per exact chunk
  int rows_a_p, rows_b_p;
  int tiles_m, tiles_n;
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

__device__ __forceinline__ float fmod_small(float x, float m, float inv_m) {
  float q = rintf(x * inv_m);
  return fmaf(-q, m, x);
}

template <int BN, bool kResidue>
__global__ void __launch_bounds__(kThreads, 1)
    limb_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmArgs args) {
  using C = Cfg<BN>;
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

  // Tile and modulus of this CTA (modulus-major, grouped tile raster).
  const int per_mod = args.tiles_m * args.tiles_n;
  const int l = blockIdx.x / per_mod;
  const int t = blockIdx.x % per_mod;
  const int group = kGroupM * args.tiles_n;
  const int first_m = (t / group) * kGroupM;
  const int gm = min(kGroupM, args.tiles_m - first_m);
  const int tm = first_m + (t % group) % gm;
  const int tn = (t % group) / gm;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4);
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
  if (warp >= 2) {
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
      const int a_row = l * 3 * args.rows_a_p + tm * kBM;
      const int b_row = l * 3 * args.rows_b_p + tn * BN;
      int issued = 0;
      for (int kb = 0; kb < kb_total; ++kb) {
        const int s = kb % C::kStages;
        const uint32_t ph = (kb / C::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, abort_word, args.flags)) break;
        uint8_t* st = smem + s * C::kStage;
        mbar_arrive_expect_tx(&full[s], C::kStage);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          tma_load_2d(st + j * kATile, &tmA, &full[s], kb * kBKBytes, a_row + j * args.rows_a_p);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          tma_load_2d(st + 3 * kATile + j * C::kBTile, &tmB, &full[s], kb * kBKBytes, b_row + j * args.rows_b_p);
        issued = kb + 1;
      }
      if (*abort_word) {
        // Let the copies already issued land before the CTA exits.
        for (int kb = (issued > C::kStages ? issued - C::kStages : 0); kb < issued; ++kb)
          drain_wait(&full[kb % C::kStages], (kb / C::kStages) & 1, args.flags);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_fp4(BN);
      const uint32_t d1 = tbase + kColD1, d2 = tbase + kColD2;
      const uint32_t s2 = tbase + kColSf2, s26 = tbase + kColSf26;
      bool ok = true;
      for (int c = 0; c < n_chunks && ok; ++c) {
        if (c > 0) {
          if (!mbar_wait(tempty, (c - 1) & 1, abort_word, args.flags)) break;
          tc_fence_after();
        }
        const int kb0 = c * args.kb_chunk;
        const int kb1 = min(kb0 + args.kb_chunk, kb_total);
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = kb % C::kStages;
          const uint32_t ph = (kb / C::kStages) & 1;
          if (!mbar_wait(&full[s], ph, abort_word, args.flags)) {
            ok = false;
            break;
          }
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
            mma_fp4(d1, a0, b0, idesc, s2, s2, acc);
            mma_fp4(d1, a0, b1, idesc, s2, s26, 1u);
            mma_fp4(d1, a1, b0, idesc, s26, s2, 1u);
            mma_fp4(d2, a0, b2, idesc, s2, s2, acc);
            mma_fp4(d2, a1, b1, idesc, s2, s2, 1u);
            mma_fp4(d2, a2, b0, idesc, s2, s2, 1u);
            mma_fp4(d2, a1, b2, idesc, s26, s2, 1u);
            mma_fp4(d2, a2, b1, idesc, s2, s26, 1u);
            mma_fp4(d2, a2, b2, idesc, s26, s26, 1u);
          }
          tc_commit(&empty[s]);
        }
        if (ok) tc_commit(tfull);
      }
      // All MMAs issued by this thread complete before teardown.
      tc_commit(mma_done);
      drain_wait(mma_done, 0, args.flags);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int grow = tm * kBM + quarter * 32 + lane;
    const float fm = args.em.m[l], finv = args.em.inv_m[l], fw = args.em.w169[l];
    for (int c = 0; c < n_chunks; ++c) {
      if (!warp_wait(tfull, c & 1, abort_word, args.flags)) break;
      tc_fence_after();
      const bool last = (c == n_chunks - 1);
#pragma unroll 1
      for (int cc = 0; cc < BN / 16; ++cc) {
        uint32_t v1[16], v2[16], run[16];
        tmem_ld16(tbase + lane_off + kColD1 + cc * 16, v1);
        tmem_ld16(tbase + lane_off + kColD2 + cc * 16, v2);
        if (c > 0) tmem_ld16(tbase + lane_off + kColRun + cc * 16, run);
        tmem_wait_ld();
        uint32_t out[16];
        if constexpr (kResidue) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float r1 = fmod_small(__uint_as_float(v1[i]), fm, finv);
            float r2 = fmod_small(__uint_as_float(v2[i]), fm, finv);
            float v = fmaf(r2, fw, r1);
            if (c > 0) v += __uint_as_float(run[i]);
            v = fmod_small(v, fm, finv);
            v = v < 0.f ? v + fm : v;
            out[i] = last ? static_cast<uint32_t>(__float2int_rn(v)) : __float_as_uint(v);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            int v = __float2int_rn(__uint_as_float(v1[i])) + 169 * __float2int_rn(__uint_as_float(v2[i]));
            if (c > 0) v += static_cast<int>(run[i]);
            out[i] = static_cast<uint32_t>(v);
          }
        }
        if (!last) {
          tmem_st16(tbase + lane_off + kColRun + cc * 16, out);
        } else if (grow < args.m) {
          const int gcol = tn * BN + cc * 16;
          if constexpr (kResidue) {
            if (gcol < args.ldr) {
              uint4 w;
              w.x = out[0] | (out[1] << 8) | (out[2] << 16) | (out[3] << 24);
              w.y = out[4] | (out[5] << 8) | (out[6] << 16) | (out[7] << 24);
              w.z = out[8] | (out[9] << 8) | (out[10] << 16) | (out[11] << 24);
              w.w = out[12] | (out[13] << 8) | (out[14] << 16) | (out[15] << 24);
              *reinterpret_cast<uint4*>(args.res_out + (static_cast<long long>(l) * args.m + grow) * args.ldr +
                                        gcol) = w;
            }
          } else {
            int32_t* crow = args.c32 + static_cast<long long>(grow) * args.ldc;
            const bool vec = ((args.ldc & 3) == 0) && ((reinterpret_cast<uintptr_t>(args.c32) & 15u) == 0) &&
                             (gcol + 16 <= args.n);
            if (vec) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<int4*>(crow + gcol + 4 * q) =
                    make_int4(static_cast<int>(out[4 * q]), static_cast<int>(out[4 * q + 1]),
                              static_cast<int>(out[4 * q + 2]), static_cast<int>(out[4 * q + 3]));
            } else {
              for (int i = 0; i < 16; ++i)
                if (gcol + i < args.n) crow[gcol + i] = static_cast<int32_t>(out[i]);
            }
          }
        }
      }
      if (!last) {
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
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

// 2-D map over a stack of limb planes: x = byte within a row, y = plane row.
bool make_plane_map(CUtensorMap* map, const uint8_t* base, int k_p, long long total_rows, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(k_p / 2), static_cast<cuuint64_t>(total_rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(k_p / 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, bool kResidue>
cudaError_t launch_bn(const LimbGemmCall& c, cudaStream_t stream) {
  using Cf = Cfg<BN>;
  const int rows_a_p = round_up(c.m, kRowAlign), rows_b_p = round_up(c.n, kRowAlign);
  const int k_p = round_up(c.k, kKAlign);
  const int r = c.residue_mode ? c.r : 1;
  CUtensorMap ma, mb;
  if (!make_plane_map(&ma, c.a_planes, k_p, 3LL * r * rows_a_p, kBM)) return cudaErrorInvalidValue;
  if (!make_plane_map(&mb, c.b_planes, k_p, 3LL * r * rows_b_p, BN)) return cudaErrorInvalidValue;
  GemmArgs a;
  a.m = c.m;
  a.n = c.n;
  a.kb_total = k_p / 128;
  a.kb_chunk = c.kc_blocks;
  a.rows_a_p = rows_a_p;
  a.rows_b_p = rows_b_p;
  a.tiles_m = (c.m + kBM - 1) / kBM;
  a.tiles_n = (c.n + BN - 1) / BN;
  a.em = c.em;
  a.res_out = c.res_out;
  a.ldr = c.ldr;
  a.c32 = c.c32;
  a.ldc = c.ldc;
  a.flags = c.flags;
  auto kern = limb_gemm_kernel<BN, kResidue>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::kSmem);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(r) * a.tiles_m * a.tiles_n;
  kern<<<static_cast<unsigned>(grid), kThreads, Cf::kSmem, stream>>>(ma, mb, a);
  return cudaGetLastError();
}

template <bool kResidue>
cudaError_t launch_mode(const LimbGemmCall& c, cudaStream_t stream) {
  if (c.n <= 16) return launch_bn<16, kResidue>(c, stream);
  if (c.n <= 32) return launch_bn<32, kResidue>(c, stream);
  if (c.n <= 64) return launch_bn<64, kResidue>(c, stream);
  return launch_bn<128, kResidue>(c, stream);
}

}  // namespace

cudaError_t launch_limb_gemm(const LimbGemmCall& call, cudaStream_t stream) {
  return call.residue_mode ? launch_mode<true>(call, stream) : launch_mode<false>(call, stream);
}

}  // namespace ozemu
