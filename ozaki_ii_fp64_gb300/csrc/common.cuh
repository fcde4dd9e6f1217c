// Shared device helpers for the ozemu kernels (sm_103a only).
//
// Inline PTX wrappers for mbarrier, TMA (cp.async.bulk.tensor), tcgen05
// (TMEM alloc / MMA / ld / st / commit) and the per-call constant blocks that
// the host passes to the kernels by value.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ozemu {

constexpr int kMaxModuli = 16;   // r limit of the three-limb and two-limb moduli
constexpr int kMaxModuliMix = 20;  // r limit of the mixed-digit moduli
constexpr int kMaxR = 20;        // size of the per-modulus constant arrays
constexpr int kRowAlign = 128;   // plane rows padded to this (GEMM tile M)
constexpr int kKAlign = 128;     // plane k padded to this (GEMM stage K)

// Device flag bits (per-device word, reported by ozemu_get_status).
constexpr uint32_t kFlagNonFinite = 1u;
constexpr uint32_t kFlagTimeout = 2u;
constexpr uint32_t kFlagRange = 4u;  // an INT4 operand held a value outside [-8, 7]

// Time limit of one pipeline wait before the kernel gives up (ns).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// The moduli in the order they are taken: greedy pairwise-coprime integers
// counting down from 256 (r moduli = the first r).  The deconstruction kernel
// derives its per-modulus constants from this table at compile time; the host
// checks its own construction against it before a launch.
constexpr uint32_t kModulusTable[kMaxModuli] = {256, 255, 253, 251, 247, 241, 239, 233,
                                                229, 227, 223, 217, 211, 199, 197, 193};

// The two-limb moduli: greedy pairwise-coprime integers counting down from
// 113.  Their balanced residues lie in [-56, 56], where the base-13 split's
// third limb is always 0, so two limbs (4 FP4 products per modulus) suffice.
constexpr uint32_t kModulusTable2[kMaxModuli] = {113, 112, 111, 109, 107, 103, 101, 97,
                                                 95,  89,  83,  79,  73,  71,  67,  61};

// The mixed-digit moduli.  The first kMixSingle are the moduli m for which
// a single member of S lies in every residue class (m <= 13; the set with the
// largest product, 8 13 11 9 7 5 = 360360, the even one first): their residue
// product is ONE FP4 product.  The rest are the greedy pairwise-coprime
// integers counting down from 113 that are coprime to those (all prime):
// two base-13 digits each, 4 FP4 products, as the two-limb moduli.
constexpr int kMixSingle = 6;
constexpr uint32_t kModulusTableMix[kMaxModuliMix] = {8,   13,  11,  9,   7,  5,  113, 109, 107, 103,
                                                      101, 97,  89,  83,  79, 73, 71,  67,  61,  59};

// Moduli of a deconstruction launch: limbs 3 takes kModulusTable, limbs 2
// kModulusTable2, limbs 1 the mixed-digit kModulusTableMix (r = 0 if the
// host's moduli differ from the table; the launch then refuses).
struct SplitModuli {
  int r;
  int limbs;
  uint32_t m[kMaxR];
};

// Per-modulus constants for the fused narrow-N path.
struct NarrowModuli {
  int r;
  uint32_t m[kMaxModuli];
  uint32_t c21[kMaxModuli];    // 2^21 mod m
  uint32_t c42[kMaxModuli];    // 2^42 mod m
  uint32_t off62[kMaxModuli];  // 2^62 mod m
  uint32_t offA[kMaxModuli];   // 2^(p_A) mod m
  uint32_t w16[kMaxModuli][4]; // 2^(16 c) mod m
};

// INT4 x INT8 in four FP4 products ([AWE] abstract): a b = sum_k g_k u_k(a)
// v_k(b) with u, v in S, the B planes on the relation sum_k t_k g_k v_k = 0
// (t = (-12, -9, -6, 3/2), kept doubled to stay integral) and
// u_k(a) = a + t_k z(a).  The codes of value i - 128: the e2m1 nibble of
// plane j's digit / 2 in byte j; 0xFFFFFFFF marks a value outside the
// operand's range.
constexpr int kFourWeights[4] = {3, 2, 6, 12};
constexpr int kFourRelation2[4] = {-24, -18, -12, 3};
struct FourCodes {
  uint32_t code[256];
};

// Per-modulus constants for the GEMM epilogue.
struct EpiModuli {
  float m[kMaxR];
  float inv_m[kMaxR];      // 1/m rounded to fp32
  float w169[kMaxR];       // 169 mod m, balanced: |w| <= m/2
};

// Mixed-radix CRT constants.
// Bit length of M = m_1 ... m_r for the moduli table (greedy pairwise-coprime
// integers from 256 down), r = 0..16; the host checks it against the table.
constexpr int kCrtBits[kMaxModuli + 1] = {0, 9, 16, 24, 32, 40, 48, 56, 64, 72, 80, 88, 95, 103, 111, 118, 126};
// The same for the two-limb moduli (kModulusTable2).
constexpr int kCrtBits2[kMaxModuli + 1] = {0, 7, 14, 21, 28, 34, 41, 48, 54, 61, 67, 74, 80, 86, 92, 99, 104};
// The same for the mixed-digit moduli (kModulusTableMix).
constexpr int kCrtBitsMix[kMaxModuliMix + 1] = {0,  4,  7,  11, 14, 17, 19, 26, 33, 39, 46,
                                                53, 59, 66, 72, 78, 85, 91, 97, 103, 109};

struct CrtModuli {
  int r;
  int limbs;                              // 3: kModulusTable, 2: kModulusTable2, 1: kModulusTableMix
  uint32_t m[kMaxR];
  uint32_t magic[kMaxR];                  // floor(2^32 / m)
  uint32_t inv[kMaxR];                    // (m_0 ... m_{l-1})^-1 mod m_l
  uint32_t g[kMaxR][kMaxR];               // g[l][j] = (m_0...m_{j-1}) inv_l mod m_l, j < l
  // Direct form: C' = sum_l c_l W_l - q M with W_l = (M/m_l) ((M/m_l)^-1 mod m_l).
  // w16[q][t][h]: 16-bit limb t of W_{4q+2h} (low half) and of W_{4q+2h+1}
  // (high half), the operands of the two-way dot products.
  uint32_t w16[5][8][2];
  uint32_t wl16[8];                       // W_{r-1} in 16-bit limbs (a lone last modulus, r = 1 mod 4)
  uint32_t m16[9];                        // M in 16-bit limbs
  float gt[9];                            // 2^(16 t) / M
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the same condition.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, at most limit_ns
// (kWaitLimitNs in the kernels; the wait probe passes a short limit).
// On time-out sets the device timeout flag and the CTA's abort word and
// returns false.  Also returns false early once another role of this CTA, or
// any CTA on the device, has timed out (the flag word is device-wide).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_word,
                                          uint32_t* flags, uint64_t limit_ns = kWaitLimitNs) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u) {
      if (*abort_word || (*reinterpret_cast<volatile uint32_t*>(flags) & kFlagTimeout)) {
        *abort_word = 1;
        return false;
      }
      uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        atomicOr(flags, kFlagTimeout);
        *abort_word = 1;
        return false;
      }
    }
  }
}

// ----------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(p)), "r"(rank));
  return out;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
               "r"(bytes)
               : "memory");
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of either CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster_addr, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1)
      : "memory");
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Pair (2-SM) forms: allocation, MMA issued by the pair's first CTA, and a
// commit that arrives on the same barrier in both CTAs.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* holder, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
#define OZEMU_MMA_FP4_PAIR(NAME, SUFFIX)                                                                         \
  __device__ __forceinline__ void NAME(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,      \
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {            \
    asm volatile(                                                                                               \
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"                                                          \
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X" SUFFIX                             \
        " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d_tmem),                                                  \
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)                     \
        : "memory");                                                                                            \
  }
OZEMU_MMA_FP4_PAIR(mma_fp4_pair, "")
OZEMU_MMA_FP4_PAIR(mma_fp4_pair_fill, ".collector::a::fill")
OZEMU_MMA_FP4_PAIR(mma_fp4_pair_use, ".collector::a::use")
OZEMU_MMA_FP4_PAIR(mma_fp4_pair_lastuse, ".collector::a::lastuse")
#undef OZEMU_MMA_FP4_PAIR

// Block-scaled FP4 MMA, NVFP4 form: A, B e2m1 from shared-memory
// descriptors, one UE4M3 scale per 16 K-elements read from TMEM.
__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Same MMA with the A-operand collector buffer: `fill` reads A from shared
// memory and keeps it, `use` reads the kept A, `lastuse` reads it and frees
// the buffer.  Consecutive products with the same A tile then read it once.
#define OZEMU_MMA_FP4_COLLECTOR(NAME, USAGE)                                                                    \
  __device__ __forceinline__ void NAME(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,      \
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {            \
    asm volatile(                                                                                               \
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"                                                          \
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X.collector::a::" USAGE               \
        " [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d_tmem),                                                  \
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)                     \
        : "memory");                                                                                            \
  }
OZEMU_MMA_FP4_COLLECTOR(mma_fp4_fill, "fill")
OZEMU_MMA_FP4_COLLECTOR(mma_fp4_use, "use")
OZEMU_MMA_FP4_COLLECTOR(mma_fp4_lastuse, "lastuse")
#undef OZEMU_MMA_FP4_COLLECTOR

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// tcgen05.wait::ld that also takes the registers of the outstanding loads
// as operands, so that no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&a)[16], uint32_t (&b)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]),
        "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
        "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&a)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x N columns of 32-bit words: register i holds column i of the
// calling thread's lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile whose rows are
// 64 bytes (128 FP4 elements) written by TMA with 64-byte swizzling: 8-row
// core groups 512 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1u) << 16;                 // leading byte offset (unused for swizzled K-major)
  d |= static_cast<uint64_t>(512u >> 4) << 32;          // stride byte offset
  d |= static_cast<uint64_t>(1u) << 46;                 // version
  d |= static_cast<uint64_t>(4u) << 61;                 // 64-byte swizzle
  return d;
}

// Instruction descriptor: kind::mxf4nvf4, A and B e2m1, K-major, UE4M3
// scales, M = m (128 for one CTA, 256 for a CTA pair), N = n.
__host__ __device__ constexpr uint32_t idesc_fp4(int n, int m = 128) {
  return (1u << 7)                                // A format: e2m1
         | (1u << 10)                             // B format: e2m1
         | (static_cast<uint32_t>(n >> 3) << 17)  // N / 8
         | (0u << 23)                             // scale type UE4M3
         | (static_cast<uint32_t>(m >> 4) << 24);    // M / 16
}

}  // namespace ozemu
