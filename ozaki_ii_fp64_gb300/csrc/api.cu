// C ABI of libozemu.so: argument checks, per-call constants, the cached
// per-device workspace and status flags, and the staging of the kernels.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <numeric>
#include <utility>
#include <vector>

#include "../../include/ozemu.h"
#include "common.cuh"
#include "kernels.h"

namespace ozemu {
namespace {

typedef unsigned __int128 u128;

// ------------------------------------------------------------------ moduli
// Greedy pairwise-coprime integers counting down from the ceiling: 256 for
// the 3-limb moduli, 113 for the two-limb moduli.  The mixed-digit list
// starts from the given single-digit moduli and continues the greedy count
// from 113 with integers coprime to every modulus taken.
uint32_t gcd_u32(uint32_t a, uint32_t b) {
  while (b) {
    uint32_t t = a % b;
    a = b;
    b = t;
  }
  return a;
}

struct ModuliTable {
  uint32_t m[kMaxR] = {};
  int count = 0;
  ModuliTable(uint32_t ceiling, int max_r, const uint32_t* first = nullptr, int n_first = 0) {
    for (int i = 0; i < n_first; ++i) m[count++] = first[i];
    for (uint32_t c = ceiling; count < max_r && c >= 2; --c) {
      bool ok = true;
      for (int j = 0; j < count && ok; ++j) ok = gcd_u32(c, m[j]) == 1;
      if (ok) m[count++] = c;
    }
  }
};

// The moduli m <= 13 whose every residue class holds a member of S (one FP4
// digit per residue), as a pairwise-coprime set of largest product, the even
// one first: their residue products take one FP4 product each.
constexpr uint32_t kSingleDigitModuli[kMixSingle] = {8, 13, 11, 9, 7, 5};

// limbs: 3 (three-limb list), 2 (two-limb list), 1 (mixed-digit list).
const ModuliTable& moduli(int limbs = 3) {
  static const ModuliTable t3(256, kMaxModuli), t2(113, kMaxModuli),
      t1(113, kMaxModuliMix, kSingleDigitModuli, kMixSingle);
  return limbs == 1 ? t1 : (limbs == 2 ? t2 : t3);
}

int max_r(int limbs) { return limbs == 1 ? kMaxModuliMix : kMaxModuli; }

// Single-digit moduli among the first r of the list (mixed-digit list only).
int single_count(int r, int limbs) { return limbs == 1 ? (r < kMixSingle ? r : kMixSingle) : 0; }

u128 modulus_product(int r, int limbs = 3) {
  u128 p = 1;
  for (int l = 0; l < r; ++l) p *= moduli(limbs).m[l];
  return p;
}

// Largest P with 2 k 2^P < M; -1 if none.
int budget_P(long long k, int r, int limbs = 3) {
  const u128 M = modulus_product(r, limbs);
  const u128 two_k = static_cast<u128>(2) * static_cast<u128>(k);
  if (!(two_k < M)) return -1;
  int P = 0;
  while (P < 126 && (two_k << (P + 1)) < M) ++P;
  return P;
}

uint32_t pow_mod(uint64_t base, uint64_t e, uint32_t m) {
  uint64_t r = 1 % m;
  base %= m;
  while (e) {
    if (e & 1) r = r * base % m;
    base = base * base % m;
    e >>= 1;
  }
  return static_cast<uint32_t>(r);
}

uint32_t inv_mod(uint32_t a, uint32_t m) {  // a coprime to m
  long long t = 0, nt = 1, rr = m, nr = a % m;
  while (nr) {
    long long q = rr / nr, x = t - q * nt;
    t = nt;
    nt = x;
    x = rr - q * nr;
    rr = nr;
    nr = x;
  }
  return static_cast<uint32_t>(t < 0 ? t + m : t);
}

SplitModuli split_moduli(int r, int limbs = 3) {
  SplitModuli s;
  std::memset(&s, 0, sizeof(s));
  s.r = r;
  s.limbs = limbs;
  for (int l = 0; l < r; ++l) {
    s.m[l] = moduli(limbs).m[l];
    const uint32_t want = limbs == 1 ? kModulusTableMix[l] : (limbs == 2 ? kModulusTable2[l] : kModulusTable[l]);
    if (s.m[l] != want) s.r = 0;  // mismatch: the launch refuses
  }
  return s;
}

NarrowModuli narrow_moduli(int r, int pA) {
  NarrowModuli nm;
  std::memset(&nm, 0, sizeof(nm));
  nm.r = r;
  for (int l = 0; l < r; ++l) {
    const uint32_t m = moduli().m[l];
    nm.m[l] = m;
    nm.c21[l] = pow_mod(2, 21, m);
    nm.c42[l] = pow_mod(2, 42, m);
    nm.off62[l] = pow_mod(2, 62, m);
    nm.offA[l] = pow_mod(2, static_cast<uint64_t>(pA), m);
    for (int c = 0; c < 4; ++c) nm.w16[l][c] = pow_mod(2, 16ull * c, m);
  }
  return nm;
}

// The fused narrow-N path is used for n <= kNarrowMaxN unless OZEMU_NARROW=0.
bool narrow_enabled() {
  const char* s = std::getenv("OZEMU_NARROW");
  return !(s && s[0] == '0');
}

// Epilogue constants of moduli first .. first + r - 1 of the list.
EpiModuli epi_moduli(int r, int limbs = 3, int first = 0) {
  EpiModuli e;
  std::memset(&e, 0, sizeof(e));
  for (int l = 0; l < r; ++l) {
    const uint32_t m = moduli(limbs).m[first + l];
    e.m[l] = static_cast<float>(m);
    e.inv_m[l] = 1.0f / static_cast<float>(m);
    const int w = static_cast<int>(169u % m);
    e.w169[l] = static_cast<float>(w > static_cast<int>(m / 2) ? w - static_cast<int>(m) : w);  // balanced
  }
  return e;
}

CrtModuli crt_moduli(int r, int limbs = 3) {
  CrtModuli c;
  std::memset(&c, 0, sizeof(c));
  c.r = r;
  c.limbs = limbs;
  u128 pref = 1;
  for (int l = 0; l < r; ++l) {
    const uint32_t m = moduli(limbs).m[l];
    c.m[l] = m;
    c.magic[l] = static_cast<uint32_t>((1ull << 32) / m);
    const uint32_t inv = inv_mod(static_cast<uint32_t>(pref % m), m);
    c.inv[l] = inv;
    u128 pj = 1;
    for (int j = 0; j < l; ++j) {
      c.g[l][j] = static_cast<uint32_t>((static_cast<uint64_t>(pj % m) * inv) % m);
      pj *= moduli(limbs).m[j];
    }
    pref *= m;
  }
  // Direct form.  pref is now M (< 2^126).
  const u128 M = pref;
  for (int l = 0; l < r; ++l) {
    const uint32_t m = moduli(limbs).m[l];
    const u128 Ml = M / m;
    const u128 W = Ml * inv_mod(static_cast<uint32_t>(Ml % m), m);  // < M
    for (int t = 0; t < 8; ++t)
      c.w16[l / 4][t][(l % 4) / 2] |= static_cast<uint32_t>((W >> (16 * t)) & 0xFFFF) << (16 * (l % 2));
    if (l == r - 1)
      for (int t = 0; t < 8; ++t) c.wl16[t] = static_cast<uint32_t>((W >> (16 * t)) & 0xFFFF);
  }
  for (int t = 0; t < 9; ++t) c.m16[t] = t < 8 ? static_cast<uint32_t>((M >> (16 * t)) & 0xFFFF) : 0u;
  int bits = 0;
  while (bits < 128 && (M >> bits) != 0) ++bits;
  const int want = limbs == 1 ? kCrtBitsMix[r] : (limbs == 2 ? kCrtBits2[r] : kCrtBits[r]);
  if (bits != want) c.r = 0;  // table mismatch: the launch refuses r = 0
  const long double Md = static_cast<long double>(M);
  for (int t = 0; t < 9; ++t) c.gt[t] = static_cast<float>(std::ldexp(1.0L, 16 * t) / Md);
  return c;
}

// ----------------------------------------------------------- device state
constexpr int kHostEvents = 32;
struct DeviceState {
  bool checked = false;
  bool supported = false;
  uint32_t* flags = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // Host-buffer product: a copy stream, a CRT stream and their events.
  cudaStream_t copy_stream = nullptr;
  cudaStream_t crt_stream = nullptr;
  cudaEvent_t ev[kHostEvents] = {};
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

int kchunk_blocks() {
  static int kc = [] {
    int v = 8192;
    if (const char* s = std::getenv("OZEMU_KCHUNK")) {
      int x = std::atoi(s);
      if (x >= 128 && x <= 8192 && x % 128 == 0) v = x;
    }
    return v / 128;
  }();
  return kc;
}

// Current device's state, created on first use.  Returns OZEMU_OK or an error.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OZEMU_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return OZEMU_ERR_CUDA;
    d.supported = (major == 10 && minor == 3);
    d.checked = true;
  }
  if (!d.supported) return OZEMU_ERR_UNSUPPORTED;
  if (!d.flags) {
    if (cudaMalloc(&d.flags, 256) != cudaSuccess) return OZEMU_ERR_ALLOC;
    if (cudaMemset(d.flags, 0, 256) != cudaSuccess) return OZEMU_ERR_CUDA;
  }
  *out = &d;
  return OZEMU_OK;
}

// Caller-set cap on each device's cached workspace (0: none).
size_t g_ws_limit = 0;

// Workspace of at least `bytes` on the current device (grows; synchronises
// the device when it has to replace a smaller buffer).  A request above the
// cap fails with OZEMU_ERR_ALLOC before anything is allocated.
int workspace(DeviceState* d, size_t bytes, uint8_t** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_ws_limit != 0 && bytes > g_ws_limit) return OZEMU_ERR_ALLOC;
  if (bytes > d->ws_bytes) {
    if (d->ws) {
      cudaDeviceSynchronize();
      cudaFree(d->ws);
      d->ws = nullptr;
      d->ws_bytes = 0;
    }
    size_t want = bytes + bytes / 8;
    if (g_ws_limit != 0 && want > g_ws_limit) want = g_ws_limit;
    if (cudaMalloc(&d->ws, want) != cudaSuccess) {
      cudaGetLastError();
      return OZEMU_ERR_ALLOC;
    }
    d->ws_bytes = want;
  }
  *out = static_cast<uint8_t*>(d->ws);
  return OZEMU_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Digit planes of the first r moduli: limbs per modulus for the three- and
// two-limb lists; one per single-digit and two per two-digit modulus for the
// mixed-digit list.
long long digit_planes(int r, int limbs) {
  if (limbs != 1) return static_cast<long long>(limbs) * r;
  const int single = single_count(r, limbs);
  return single + 2LL * (r - single);
}

size_t plane_bytes(long long rows, long long k, int r, int limbs = 3) {
  return static_cast<size_t>(digit_planes(r, limbs) * round_up(static_cast<int>(rows), kRowAlign)) *
         static_cast<size_t>(round_up(static_cast<int>(k), kKAlign) / 2);
}

bool rows_ok(int rows, int r) {  // plane-row coordinates fit in int
  return 3LL * r * round_up(rows, kRowAlign) < (1LL << 31);
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? OZEMU_OK : OZEMU_ERR_CUDA; }

// ---------------------------------------------------------------- stages
int split_rows_f64(int rows, int k, const double* X, long long ldx, int p, int r, uint8_t* planes,
                   int32_t* shifts, DeviceState* d, cudaStream_t st, int limbs = 3) {
  return cuda_status(
      launch_split_rows_f64(X, ldx, rows, k, p, split_moduli(r, limbs), planes, shifts, d->flags, st));
}

// Columns of X (k x cols) into limb planes, without a transposed copy:
// scratch holds the cols column maxima (8 bytes each).
int split_cols_f64(int k, int cols, const double* X, long long ldx, int p, int r, uint8_t* planes,
                   int32_t* shifts, void* scratch, DeviceState* d, cudaStream_t st, int limbs = 3) {
  return cuda_status(launch_split_cols_f64(X, ldx, k, cols, p, split_moduli(r, limbs), planes, shifts,
                                           static_cast<unsigned long long*>(scratch), d->flags, st));
}

// Bytes of the column-maximum scratch of a column split of `cols` columns.
size_t colmax_bytes(int cols) { return align256(static_cast<size_t>(cols > 0 ? cols : 1) * 8); }

int residue_gemm(int m, int n, int k, int r, const uint8_t* ap, const uint8_t* bp, uint8_t* res, DeviceState* d,
                 cudaStream_t st, int limbs = 3) {
  if (limbs == 1) {
    // Mixed-digit list: the single-digit moduli (one FP4 product each) and
    // the two-digit moduli (four) are two launches over their own planes,
    // writing consecutive moduli of the residue output.
    const int single = single_count(r, limbs);
    const size_t kp2 = static_cast<size_t>(round_up(k, kKAlign) / 2);
    const size_t a_off = static_cast<size_t>(single) * round_up(m, kRowAlign) * kp2;
    const size_t b_off = static_cast<size_t>(single) * round_up(n, kRowAlign) * kp2;
    const size_t r_off = static_cast<size_t>(single) * m * round_up(n, 16);
    for (int grp = 0; grp < 2; ++grp) {
      const int rg = grp == 0 ? single : r - single;
      if (rg == 0) continue;
      LimbGemmCall c;
      c.residue_mode = true;
      c.m = m;
      c.n = n;
      c.k = k;
      c.r = rg;
      c.a_planes = grp == 0 ? ap : ap + a_off;
      c.b_planes = grp == 0 ? bp : bp + b_off;
      c.res_out = grp == 0 ? res : res + r_off;
      c.ldr = round_up(n, 16);
      c.c32 = nullptr;
      c.ldc = 0;
      c.kc_blocks = kchunk_blocks();
      c.limbs = grp == 0 ? 1 : 2;
      c.em = epi_moduli(rg, limbs, grp == 0 ? 0 : single);
      c.flags = d->flags;
      const int s = cuda_status(launch_limb_gemm(c, st));
      if (s != OZEMU_OK) return s;
    }
    return OZEMU_OK;
  }
  LimbGemmCall c;
  c.residue_mode = true;
  c.m = m;
  c.n = n;
  c.k = k;
  c.r = r;
  c.a_planes = ap;
  c.b_planes = bp;
  c.res_out = res;
  c.ldr = round_up(n, 16);
  c.c32 = nullptr;
  c.ldc = 0;
  c.kc_blocks = kchunk_blocks();
  c.limbs = limbs;
  c.em = epi_moduli(r, limbs);
  c.flags = d->flags;
  return cuda_status(launch_limb_gemm(c, st));
}

// Residues and shifts of C' = A'B' for n <= kNarrowMaxN: B's column
// residues, then the fused pass over A's rows.  Same bytes as the
// limb-plane path.
int narrow_residues(int m, int n, int k, const double* A, long long lda, const double* B, long long ldb, int r,
                    int pa_bits, int pb_bits, uint8_t* res, int32_t* sa, int32_t* sb, DeviceState* d,
                    cudaStream_t st) {
  NarrowCall c;
  c.m = m;
  c.n = n;
  c.k = k;
  c.kp = round_up(k, 16);
  c.pA = pa_bits;
  c.pB = pb_bits;
  c.A = A;
  c.lda = lda;
  c.B = B;
  c.ldb = ldb;
  c.nm = narrow_moduli(r, pa_bits);
  c.ldr = round_up(n, 16);
  const size_t bres = align256(static_cast<size_t>(n) * r * c.kp);
  const size_t cs = align256(static_cast<size_t>(n) * r * 4);
  uint8_t* ws = nullptr;
  int s = workspace(d, bres + cs, &ws);
  if (s != OZEMU_OK) return s;
  c.bres = ws;
  c.colsum = reinterpret_cast<int32_t*>(ws + bres);
  c.res = res;
  c.sa = sa;
  c.sb = sb;
  c.flags = d->flags;
  return cuda_status(launch_narrow_residues(c, st));
}

// C = A B for n <= kNarrowMaxN through narrow_residues and the CRT.
int dgemm_narrow(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc, int r,
                 int pa_bits, int pb_bits, DeviceState* d, cudaStream_t st) {
  const size_t bres = align256(static_cast<size_t>(n) * r * round_up(k, 16));
  const size_t cs = align256(static_cast<size_t>(n) * r * 4);
  const size_t rb = align256(ozemu_residue_bytes(m, n, r));
  const size_t sa = align256(static_cast<size_t>(m) * 4), sb = align256(static_cast<size_t>(n) * 4);
  uint8_t* ws = nullptr;
  int s = workspace(d, bres + cs + rb + sa + sb, &ws);
  if (s != OZEMU_OK) return s;
  // narrow_residues takes the front of the same workspace for B's residues.
  uint8_t* res = ws + bres + cs;
  int32_t* sap = reinterpret_cast<int32_t*>(res + rb);
  int32_t* sbp = reinterpret_cast<int32_t*>(res + rb + sa);
  s = narrow_residues(m, n, k, A, lda, B, ldb, r, pa_bits, pb_bits, res, sap, sbp, d, st);
  if (s != OZEMU_OK) return s;
  return cuda_status(launch_crt_f64(m, n, res, round_up(n, 16), sap, sbp, C, ldc, crt_moduli(r), st));
}

// Streams and events of the host-buffer product, created on first use.
int pipeline_state(DeviceState* d) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (d->copy_stream) return OZEMU_OK;
  if (cudaStreamCreateWithFlags(&d->copy_stream, cudaStreamNonBlocking) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (cudaStreamCreateWithFlags(&d->crt_stream, cudaStreamNonBlocking) != cudaSuccess) return OZEMU_ERR_CUDA;
  for (int i = 0; i < kHostEvents; ++i)
    if (cudaEventCreateWithFlags(&d->ev[i], cudaEventDisableTiming) != cudaSuccess) return OZEMU_ERR_CUDA;
  return OZEMU_OK;
}

// C = A B over row chunks of A, each an independent product A_c B, pipelined
// on the caller's stream and two helper streams.  With host buffers
// (from_host): the copy stream brings B in, then A_0, A_1, ...; the caller's
// stream splits B's columns, then per chunk splits its rows and runs the limb
// GEMM; the CRT stream runs each chunk's CRT beside the next chunk's GEMM;
// the copy stream sends each chunk of C out as soon as it is ready.  With
// device buffers the helper stream splits the chunks' rows ahead of the GEMMs
// instead.  The caller's stream completes after the last CRT (device) or
// copy out (host); the helper streams start after everything the caller
// queued before.
constexpr int kMaxChunks = 8;

int dgemm_chunked(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc, int r,
                  int pa_bits, int pb_bits, bool from_host, DeviceState* d, cudaStream_t stream, int limbs = 3) {
  int s = pipeline_state(d);
  if (s != OZEMU_OK) return s;
  // Row chunks of A: up to four equal chunks; with host operands and
  // m >= 4096 the first two are half as tall (m/8), so that the first
  // products start early and the later ones run at full size.
  int row0s[kMaxChunks + 1];
  int nch = 0;
  if (from_host && m >= 4096) {
    const int base = round_up((m + 7) / 8, 256);
    for (int row = 0; row < m; row += (nch < 2 ? base : 2 * base)) row0s[nch++] = row;
  } else {
    const int step = m >= 2048 ? round_up((m + 3) / 4, 256) : m;
    for (int row = 0; row < m; row += step) row0s[nch++] = row;
  }
  row0s[nch] = m;
  int chunk = 0;  // tallest chunk (sizes the per-chunk buffers)
  for (int c = 0; c < nch; ++c) chunk = row0s[c + 1] - row0s[c] > chunk ? row0s[c + 1] - row0s[c] : chunk;
  // With host operands B comes over in two blocks of columns, so that the
  // first products start once its first block is in and split.  The first
  // block is a whole number of pair tiles (224 columns), so that the split
  // adds no partially filled tile column.
  const int bsplit = (from_host && n >= 4096) ? (n / 2) / kPairTileCols * kPairTileCols : n;
  const int nbc = bsplit < n ? 2 : 1;
  const int bcols = nbc > 1 && n - bsplit > bsplit ? n - bsplit : bsplit;  // widest block (sizes the buffers)
  const size_t szA = from_host ? align256(static_cast<size_t>(m) * k * 8) : 0;
  const size_t szB = from_host ? align256(static_cast<size_t>(k) * n * 8) : 0;
  const size_t szC = from_host ? align256(static_cast<size_t>(m) * n * 8) : 0;
  const size_t szBt = colmax_bytes(bcols);
  const size_t szBp = align256(plane_bytes(bcols, k, r, limbs)), szSb = align256(static_cast<size_t>(bcols) * 4);
  const size_t szAp = align256(plane_bytes(chunk, k, r, limbs)), szSa = align256(static_cast<size_t>(chunk) * 4);
  const size_t szRes = align256(ozemu_residue_bytes(chunk, bcols, r));
  uint8_t* buf = nullptr;
  s = workspace(d, szA + szB + szC + szBt + nbc * (szBp + szSb) + nch * (szAp + szSa + nbc * szRes), &buf);
  if (s != OZEMU_OK) return s;
  // Operands on the device: copies in the workspace, or the caller's buffers.
  const double* Ad = from_host ? reinterpret_cast<const double*>(buf) : A;
  const double* Bd = from_host ? reinterpret_cast<const double*>(buf + szA) : B;
  double* Cd = from_host ? reinterpret_cast<double*>(buf + szA + szB) : C;
  const long long ldad = from_host ? k : lda, ldbd = from_host ? n : ldb, ldcd = from_host ? n : ldc;
  void* Bt = buf + szA + szB + szC;  // column maxima of B's split
  uint8_t* per_bblock = buf + szA + szB + szC + szBt;           // [nbc] planes + shifts of B's column blocks
  uint8_t* per_chunk = per_bblock + nbc * (szBp + szSb);       // [nch] planes + shifts of A's rows, residues
  cudaStream_t cs = d->copy_stream, xs = d->crt_stream;
  cudaEvent_t* ev = d->ev;
  constexpr int evStart = 0, evB = 1, evA = 3, evG = 3 + kMaxChunks, evC = evG + 1, evD = evC + 1;  // nbc <= 2
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  const CrtModuli cm = crt_moduli(r, limbs);
  auto bcol0 = [&](int j) { return j == 0 ? 0 : bsplit; };
  auto bwidth = [&](int j) { return j == 0 ? bsplit : n - bsplit; };
  auto bplanes = [&](int j) { return per_bblock + j * (szBp + szSb); };
  auto bshifts = [&](int j) { return reinterpret_cast<int32_t*>(per_bblock + j * (szBp + szSb) + szBp); };
  auto copy_b = [&](int j) {
    return cudaMemcpy2DAsync(const_cast<double*>(Bd) + bcol0(j), static_cast<size_t>(n) * 8, B + bcol0(j),
                             static_cast<size_t>(ldb) * 8, static_cast<size_t>(bwidth(j)) * 8, k, h2d, cs) ==
                   cudaSuccess &&
           cudaEventRecord(ev[evB + j], cs) == cudaSuccess;
  };
  auto split_b = [&](int j) -> int {
    if (from_host && cudaStreamWaitEvent(stream, ev[evB + j], 0) != cudaSuccess) return OZEMU_ERR_CUDA;
    return split_cols_f64(k, bwidth(j), Bd + bcol0(j), ldbd, pb_bits, r, bplanes(j), bshifts(j), Bt, d, stream,
                          limbs);
  };
  if (cudaEventRecord(ev[evStart], stream) != cudaSuccess || cudaStreamWaitEvent(cs, ev[evStart], 0) != cudaSuccess ||
      cudaStreamWaitEvent(xs, ev[evStart], 0) != cudaSuccess)
    return OZEMU_ERR_CUDA;
  // Copy stream: B's first block, the first nfirst row chunks of A, B's other
  // block, A's other rows (device operands: the splits of A's rows).  The
  // products of the first chunks with B's first block keep the GPU busy
  // while B's second block comes over.
  int nfirst = nch;  // chunks that cover at least half of A's rows
  if (nbc > 1)
    for (nfirst = 1; nfirst < nch && 2 * row0s[nfirst] < m; ++nfirst) {
    }
  if (from_host && !copy_b(0)) return OZEMU_ERR_CUDA;
  for (int c = 0; c < nch; ++c) {
    const int row0 = row0s[c], mc = row0s[c + 1] - row0;
    if (from_host) {
      if (cudaMemcpy2DAsync(const_cast<double*>(Ad) + static_cast<size_t>(row0) * k, k * 8,
                            A + static_cast<size_t>(row0) * lda, static_cast<size_t>(lda) * 8,
                            static_cast<size_t>(k) * 8, mc, h2d, cs) != cudaSuccess)
        return OZEMU_ERR_CUDA;
    } else {
      uint8_t* ap = per_chunk + c * (szAp + szSa + nbc * szRes);
      s = split_rows_f64(mc, k, Ad + row0 * ldad, ldad, pa_bits, r, ap, reinterpret_cast<int32_t*>(ap + szAp), d, cs,
                         limbs);
      if (s != OZEMU_OK) return s;
    }
    if (cudaEventRecord(ev[evA + c], cs) != cudaSuccess) return OZEMU_ERR_CUDA;
    if (c == nfirst - 1 && from_host)
      for (int j = 1; j < nbc; ++j)
        if (!copy_b(j)) return OZEMU_ERR_CUDA;
  }
  // One (row chunk, column block) product, its CRT and its copy out.  A
  // chunk's rows are split before its first product (block 0).
  auto block = [&](int c, int j) -> int {
    const int row0 = row0s[c], mc = row0s[c + 1] - row0;
    uint8_t* ap = per_chunk + c * (szAp + szSa + nbc * szRes);
    int32_t* sap = reinterpret_cast<int32_t*>(ap + szAp);
    if (j == 0) {
      if (cudaStreamWaitEvent(stream, ev[evA + c], 0) != cudaSuccess) return OZEMU_ERR_CUDA;
      if (from_host) {
        const int st = split_rows_f64(mc, k, Ad + row0 * ldad, ldad, pa_bits, r, ap, sap, d, stream, limbs);
        if (st != OZEMU_OK) return st;
      }
    }
    const int col0 = bcol0(j), nc = bwidth(j);
    uint8_t* res = ap + szAp + szSa + j * szRes;
    const int st = residue_gemm(mc, nc, k, r, ap, bplanes(j), res, d, stream, limbs);
    if (st != OZEMU_OK) return st;
    // One event each for the product -> CRT and CRT -> copy hand-offs: each
    // record is waited on before the next one.
    if (cudaEventRecord(ev[evG], stream) != cudaSuccess || cudaStreamWaitEvent(xs, ev[evG], 0) != cudaSuccess)
      return OZEMU_ERR_CUDA;
    if (launch_crt_f64(mc, nc, res, round_up(nc, 16), sap, bshifts(j), Cd + row0 * ldcd + col0, ldcd, cm, xs) !=
            cudaSuccess ||
        cudaEventRecord(ev[evC], xs) != cudaSuccess)
      return OZEMU_ERR_CUDA;
    if (from_host) {
      if (cudaStreamWaitEvent(cs, ev[evC], 0) != cudaSuccess ||
          cudaMemcpy2DAsync(C + static_cast<size_t>(row0) * ldc + col0, static_cast<size_t>(ldc) * 8,
                            Cd + row0 * ldcd + col0, static_cast<size_t>(ldcd) * 8, static_cast<size_t>(nc) * 8, mc,
                            d2h, cs) != cudaSuccess)
        return OZEMU_ERR_CUDA;
    }
    return OZEMU_OK;
  };
  // Products: the first chunks with B's first block, then with its other
  // block, then the remaining chunks with both.
  s = split_b(0);
  if (s != OZEMU_OK) return s;
  for (int c = 0; c < nfirst; ++c)
    if ((s = block(c, 0)) != OZEMU_OK) return s;
  for (int j = 1; j < nbc; ++j) {
    if ((s = split_b(j)) != OZEMU_OK) return s;
    for (int c = 0; c < nfirst; ++c)
      if ((s = block(c, j)) != OZEMU_OK) return s;
  }
  for (int c = nfirst; c < nch; ++c)
    for (int j = 0; j < nbc; ++j)
      if ((s = block(c, j)) != OZEMU_OK) return s;
  // The caller's stream completes only after the last CRT (or copy out).
  cudaStream_t last = from_host ? cs : xs;
  if (cudaEventRecord(ev[evD], last) != cudaSuccess || cudaStreamWaitEvent(stream, ev[evD], 0) != cudaSuccess)
    return OZEMU_ERR_CUDA;
  return OZEMU_OK;
}

int limb_gemm_s32(int m, int n, int k, const uint8_t* ap, const uint8_t* bp, int32_t* C, long long ldc,
                  DeviceState* d, cudaStream_t st) {
  LimbGemmCall c;
  c.residue_mode = false;
  c.m = m;
  c.n = n;
  c.k = k;
  c.r = 1;
  c.a_planes = ap;
  c.b_planes = bp;
  c.res_out = nullptr;
  c.ldr = 0;
  c.c32 = C;
  c.ldc = ldc;
  c.kc_blocks = kchunk_blocks();
  c.em = epi_moduli(1);
  c.flags = d->flags;
  return cuda_status(launch_limb_gemm(c, st));
}

constexpr int kMaxKInt32 = 131071;

// ------------------------------------------------ INT4 x INT8, four planes
// [AWE] abstract: an INT4 x INT8 product in four FP4 products.  The encoding
// a b = sum_k g_k u_k(a) v_k(b) (weights and relation in common.cuh): the A
// planes u_k(a) = a + t_k z(a) with the smallest |z| (then the smaller z) of
// the form n/d, d in {1, 2, 3, 4, 6}, that puts every u_k in S; the B planes
// the v in S^4 on the relation with b = sum_k g_k v_k of smallest digit sum,
// then lexicographically smallest.  Built once on the host.
constexpr int kMaxKS4 = 2097151;  // |C| <= 1024 k stays below 2^31
constexpr int kDigitsS[15] = {0, 1, -1, 2, -2, 3, -3, 4, -4, 6, -6, 8, -8, 12, -12};

bool digit_in_s(int d) {
  for (int x : kDigitsS)
    if (x == d) return true;
  return false;
}

uint32_t e2m1_code_host(int d) {  // the e2m1 nibble of d / 2 for d in S
  const int a = d < 0 ? -d : d;
  const uint32_t mag = a <= 4 ? static_cast<uint32_t>(a) : (a == 6 ? 5u : (a == 8 ? 6u : 7u));
  return (d < 0 ? 8u : 0u) | mag;
}

struct FourTables {
  FourCodes a, b;
  bool ok = false;
};

FourTables build_four_tables() {
  FourTables t;
  for (int i = 0; i < 256; ++i) t.a.code[i] = t.b.code[i] = 0xFFFFFFFFu;
  // Candidates z = n / d in lowest terms, by |z| then z.
  std::vector<std::pair<int, int>> zs;
  for (int d : {1, 2, 3, 4, 6})
    for (int n = -48; n <= 48; ++n) {
      int g = std::gcd(n < 0 ? -n : n, d);
      if (g == 0) g = d;
      const std::pair<int, int> z(n / g, d / g);
      if (std::find(zs.begin(), zs.end(), z) == zs.end()) zs.push_back(z);
    }
  std::sort(zs.begin(), zs.end(), [](const std::pair<int, int>& x, const std::pair<int, int>& y) {
    const long long ax = static_cast<long long>(std::abs(x.first)) * y.second;
    const long long ay = static_cast<long long>(std::abs(y.first)) * x.second;
    if (ax != ay) return ax < ay;
    return static_cast<long long>(x.first) * y.second < static_cast<long long>(y.first) * x.second;
  });
  for (int a = -8; a <= 7; ++a) {
    bool found = false;
    for (const auto& z : zs) {
      uint32_t code = 0;
      bool ok = true;
      for (int k = 0; k < 4 && ok; ++k) {
        const int num = kFourRelation2[k] * z.first, den = 2 * z.second;  // t_k z = num / den
        if (num % den != 0) {
          ok = false;
          break;
        }
        const int u = a + num / den;
        if (!digit_in_s(u)) ok = false;
        code |= e2m1_code_host(u) << (8 * k);
      }
      if (ok) {
        t.a.code[a + 128] = code;
        found = true;
        break;
      }
    }
    if (!found) return t;
  }
  int best_sum[256];
  int best_v[256][4];
  for (int i = 0; i < 256; ++i) best_sum[i] = -1;
  for (int v0 : kDigitsS)
    for (int v1 : kDigitsS)
      for (int v2 : kDigitsS)
        for (int v3 : kDigitsS) {
          const int v[4] = {v0, v1, v2, v3};
          int rel = 0, b = 0, sum = 0;
          for (int k = 0; k < 4; ++k) {
            rel += kFourRelation2[k] * kFourWeights[k] * v[k];
            b += kFourWeights[k] * v[k];
            sum += std::abs(v[k]);
          }
          if (rel != 0 || b < -128 || b > 127) continue;
          const int i = b + 128;
          const bool better = best_sum[i] < 0 || sum < best_sum[i] ||
                              (sum == best_sum[i] && std::lexicographical_compare(v, v + 4, best_v[i], best_v[i] + 4));
          if (better) {
            best_sum[i] = sum;
            for (int k = 0; k < 4; ++k) best_v[i][k] = v[k];
          }
        }
  for (int i = 0; i < 256; ++i) {
    if (best_sum[i] < 0) return t;
    uint32_t code = 0;
    for (int k = 0; k < 4; ++k) code |= e2m1_code_host(best_v[i][k]) << (8 * k);
    t.b.code[i] = code;
  }
  t.ok = true;
  return t;
}

const FourTables& four_tables() {
  static const FourTables t = build_four_tables();
  return t;
}

size_t four_plane_bytes(int rows, int k) {
  return static_cast<size_t>(round_up(rows, kRowAlign)) * 2 * static_cast<size_t>(round_up(k, kKAlign));
}

// Scratch of the allocation-free entry point: one fixed static device array
// (its device address is looked up per device, never allocated by us).
constexpr size_t kNoAllocBytes = size_t(64) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
  bool ready = false;
  uint8_t* base = nullptr;  // device address of g_noalloc_scratch
};
NoAllocDevice g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the static scratch for the current device; the lookup
// happens once per device with that device current.
// Diagnostic of the bounded pipeline wait: one thread waits, with a short
// limit, on an mbarrier phase that nothing completes.  The wait gives up,
// sets the time-out bit of `flags` and returns; no copy or MMA is in flight.
__global__ void wait_probe_kernel(uint32_t* flags, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_word = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_word, flags, limit_ns);
  __syncthreads();
}

int noalloc_scratch(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OZEMU_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return OZEMU_ERR_CUDA;
    if (!(major == 10 && minor == 3)) return OZEMU_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return OZEMU_ERR_CUDA;
    }
    d.base = static_cast<uint8_t*>(p);
    d.ready = true;
  }
  *out = d.base;
  return OZEMU_OK;
}

}  // namespace
}  // namespace ozemu

using namespace ozemu;

extern "C" {

int ozemu_max_moduli(void) { return kMaxModuli; }

int ozemu_moduli(int r, int32_t* out) {
  if (r < 1 || r > kMaxModuli || !out) return OZEMU_ERR_INVALID_ARG;
  for (int l = 0; l < r; ++l) out[l] = static_cast<int32_t>(moduli().m[l]);
  return OZEMU_OK;
}

int ozemu_bit_budget(int k, int r, int* p_a, int* p_b) {
  if (k < 1 || r < 1 || r > kMaxModuli || !p_a || !p_b) return OZEMU_ERR_INVALID_ARG;
  const int P = budget_P(k, r);
  if (P < 0) return OZEMU_ERR_INVALID_ARG;
  *p_a = (P + 1) / 2;
  *p_b = P / 2;
  return OZEMU_OK;
}

size_t ozemu_plane_bytes(int rows, int k, int r) {
  if (rows < 0 || k < 0 || r < 1 || r > kMaxModuli) return 0;
  return plane_bytes(rows, k, r);
}

size_t ozemu_residue_bytes(int m, int n, int r) {
  if (m < 0 || n < 0 || r < 1 || r > kMaxR) return 0;
  return static_cast<size_t>(r) * static_cast<size_t>(m) * static_cast<size_t>(round_up(n, 16));
}

int ozemu_split_rows_f64(int rows, int k, const double* X, int ldx, int p, int r, uint8_t* planes,
                         int32_t* shifts, cudaStream_t stream) {
  if (rows < 0 || k < 0 || ldx < (k > 1 ? k : 1) || p < 0 || p > 62 || r < 1 || r > kMaxModuli)
    return OZEMU_ERR_INVALID_ARG;
  if (rows == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !shifts || !aligned16(planes) || !rows_ok(rows, r)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  return split_rows_f64(rows, k, X, ldx, p, r, planes, shifts, d, stream);
}

static int split_cols_entry(int k, int cols, const double* X, int ldx, int p, int r, uint8_t* planes,
                            int32_t* shifts, cudaStream_t stream, int limbs) {
  if (k < 0 || cols < 0 || ldx < (cols > 1 ? cols : 1) || p < 0 || p > 62 || r < 1 || r > max_r(limbs))
    return OZEMU_ERR_INVALID_ARG;
  if (cols == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !shifts || !aligned16(planes) || !rows_ok(cols, r)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  uint8_t* ws = nullptr;
  s = workspace(d, colmax_bytes(cols), &ws);
  if (s != OZEMU_OK) return s;
  return split_cols_f64(k, cols, X, ldx, p, r, planes, shifts, ws, d, stream, limbs);
}

int ozemu_split_cols_f64(int k, int cols, const double* X, int ldx, int p, int r, uint8_t* planes,
                         int32_t* shifts, cudaStream_t stream) {
  return split_cols_entry(k, cols, X, ldx, p, r, planes, shifts, stream, 3);
}

int ozemu_split_rows_s8(int rows, int k, const int8_t* X, int ldx, uint8_t* planes, cudaStream_t stream) {
  if (rows < 0 || k < 0 || ldx < (k > 1 ? k : 1)) return OZEMU_ERR_INVALID_ARG;
  if (rows == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !aligned16(planes) || !rows_ok(rows, 1)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  return cuda_status(launch_split_rows_s8(X, ldx, rows, k, planes, stream));
}

int ozemu_split_cols_s8(int k, int cols, const int8_t* X, int ldx, uint8_t* planes, cudaStream_t stream) {
  if (k < 0 || cols < 0 || ldx < (cols > 1 ? cols : 1)) return OZEMU_ERR_INVALID_ARG;
  if (cols == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !aligned16(planes) || !rows_ok(cols, 1)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(cudaMemsetAsync(planes, 0, plane_bytes(cols, 0, 1), stream));
  return cuda_status(launch_split_cols_s8(X, ldx, k, cols, planes, stream));
}

size_t ozemu_res8_bytes(int rows, int k, int r) {
  if (rows < 0 || k < 0 || r < 1 || r > kMaxModuli) return 0;
  return static_cast<size_t>(r) * round_up(rows, kRowAlign) * static_cast<size_t>(round_up(k, kKAlign));
}

int ozemu_split_rows_f64_res8(int rows, int k, const double* X, int ldx, int p, int r, int8_t* res8,
                              int32_t* shifts, cudaStream_t stream) {
  if (rows < 0 || k < 0 || ldx < (k > 1 ? k : 1) || p < 0 || p > 62 || r < 1 || r > kMaxModuli)
    return OZEMU_ERR_INVALID_ARG;
  if (rows == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !res8 || !shifts || !aligned16(res8) || !rows_ok(rows, r)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  return cuda_status(launch_split_rows_f64_res8(X, ldx, rows, k, p, split_moduli(r), res8, shifts, d->flags, stream));
}

int ozemu_split_cols_f64_res8(int k, int cols, const double* X, int ldx, int p, int r, int8_t* res8,
                              int32_t* shifts, cudaStream_t stream) {
  if (k < 0 || cols < 0 || ldx < (cols > 1 ? cols : 1) || p < 0 || p > 62 || r < 1 || r > kMaxModuli)
    return OZEMU_ERR_INVALID_ARG;
  if (cols == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !res8 || !shifts || !aligned16(res8) || !rows_ok(cols, r)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  uint8_t* ws = nullptr;
  s = workspace(d, align256(static_cast<size_t>(k > 0 ? k : 1) * cols * sizeof(double)), &ws);
  if (s != OZEMU_OK) return s;
  double* t = reinterpret_cast<double*>(ws);
  if (k > 0 && launch_transpose_f64(X, ldx, k, cols, t, k, stream) != cudaSuccess) return OZEMU_ERR_CUDA;
  return cuda_status(
      launch_split_rows_f64_res8(t, k > 0 ? k : 1, cols, k, p, split_moduli(r), res8, shifts, d->flags, stream));
}

int ozemu_residue_gemm_i8(int m, int n, int k, int r, const int8_t* a_res8, const int8_t* b_res8,
                          uint8_t* residues, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || r < 1 || r > kMaxModuli) return OZEMU_ERR_INVALID_ARG;
  if (k > kMaxKInt32) return OZEMU_ERR_K_OVERFLOW;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!residues || !aligned16(residues) || !rows_ok(m, r) || !rows_ok(n, r)) return OZEMU_ERR_INVALID_ARG;
  if (k > 0 && (!a_res8 || !b_res8 || !aligned16(a_res8) || !aligned16(b_res8))) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(cudaMemsetAsync(residues, 0, ozemu_residue_bytes(m, n, r), stream));
  return cuda_status(launch_residue_gemm_i8(m, n, k, r, a_res8, b_res8, residues, round_up(n, 16), epi_moduli(r),
                                            stream));
}

static int residue_gemm_entry(int m, int n, int k, int r, const uint8_t* a_planes, const uint8_t* b_planes,
                              uint8_t* residues, cudaStream_t stream, int limbs) {
  if (m < 0 || n < 0 || k < 0 || r < 1 || r > max_r(limbs)) return OZEMU_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!residues || !aligned16(residues) || !rows_ok(m, r) || !rows_ok(n, r)) return OZEMU_ERR_INVALID_ARG;
  if (k > 0 && (!a_planes || !b_planes || !aligned16(a_planes) || !aligned16(b_planes)))
    return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0)
    return cuda_status(cudaMemsetAsync(residues, 0, ozemu_residue_bytes(m, n, r), stream));
  return residue_gemm(m, n, k, r, a_planes, b_planes, residues, d, stream, limbs);
}

int ozemu_residue_gemm(int m, int n, int k, int r, const uint8_t* a_planes, const uint8_t* b_planes,
                       uint8_t* residues, cudaStream_t stream) {
  return residue_gemm_entry(m, n, k, r, a_planes, b_planes, residues, stream, 3);
}

int ozemu_limb_gemm_s32(int m, int n, int k, const uint8_t* a_planes, const uint8_t* b_planes, int32_t* C32,
                        int ldc, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || ldc < (n > 1 ? n : 1)) return OZEMU_ERR_INVALID_ARG;
  if (k > kMaxKInt32) return OZEMU_ERR_K_OVERFLOW;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C32 || !rows_ok(m, 1) || !rows_ok(n, 1)) return OZEMU_ERR_INVALID_ARG;
  if (k > 0 && (!a_planes || !b_planes || !aligned16(a_planes) || !aligned16(b_planes)))
    return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(launch_zero_s32(C32, m, n, ldc, stream));
  return limb_gemm_s32(m, n, k, a_planes, b_planes, C32, ldc, d, stream);
}

int ozemu_narrow_max_n(void) { return kNarrowMaxN; }

int ozemu_residues_narrow_f64(int m, int n, int k, int r, const double* A, int lda, const double* B, int ldb,
                              uint8_t* residues, int32_t* shifts_a, int32_t* shifts_b, cudaStream_t stream) {
  if (m < 0 || n < 1 || n > kNarrowMaxN || k < 1 || k > kNarrowMaxK || r < 1 || r > kMaxModuli)
    return OZEMU_ERR_INVALID_ARG;
  if (lda < k || ldb < n) return OZEMU_ERR_INVALID_ARG;
  if (m == 0) return OZEMU_OK;
  if (!A || !B || !residues || !aligned16(residues) || !shifts_a || !shifts_b || !rows_ok(m, r))
    return OZEMU_ERR_INVALID_ARG;
  int pa_bits = 0, pb_bits = 0;
  if (ozemu_bit_budget(k, r, &pa_bits, &pb_bits) != OZEMU_OK || pa_bits > kNarrowMaxP) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  return narrow_residues(m, n, k, A, lda, B, ldb, r, pa_bits, pb_bits, residues, shifts_a, shifts_b, d, stream);
}

static int crt_entry(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a, const int32_t* shifts_b,
                     double* C, int ldc, cudaStream_t stream, int limbs) {
  if (m < 0 || n < 0 || r < 1 || r > max_r(limbs) || ldc < (n > 1 ? n : 1)) return OZEMU_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!residues || !aligned16(residues) || !shifts_a || !shifts_b || !C) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  return cuda_status(
      launch_crt_f64(m, n, residues, round_up(n, 16), shifts_a, shifts_b, C, ldc, crt_moduli(r, limbs), stream));
}

int ozemu_crt_f64(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a, const int32_t* shifts_b,
                  double* C, int ldc, cudaStream_t stream) {
  return crt_entry(m, n, r, residues, shifts_a, shifts_b, C, ldc, stream, 3);
}

int ozemu_igemm_s8(int m, int n, int k, const int8_t* A, const int8_t* B, int32_t* C32, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0) return OZEMU_ERR_INVALID_ARG;
  if (k > kMaxKInt32) return OZEMU_ERR_K_OVERFLOW;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C32 || (k > 0 && (!A || !B)) || !rows_ok(m, 1) || !rows_ok(n, 1)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(launch_zero_s32(C32, m, n, n, stream));
  const size_t pa = align256(plane_bytes(m, k, 1)), pb = align256(plane_bytes(n, k, 1));
  uint8_t* ws = nullptr;
  s = workspace(d, pa + pb, &ws);
  if (s != OZEMU_OK) return s;
  uint8_t* ap = ws;
  uint8_t* bp = ws + pa;
  // The two splits are small and latency-bound: A's rows on a helper stream
  // beside B's columns on the caller's stream.
  s = pipeline_state(d);
  if (s != OZEMU_OK) return s;
  cudaStream_t xs = d->copy_stream;
  if (cudaEventRecord(d->ev[0], stream) != cudaSuccess || cudaStreamWaitEvent(xs, d->ev[0], 0) != cudaSuccess)
    return OZEMU_ERR_CUDA;
  if (launch_split_rows_s8(A, k, m, k, ap, xs) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (cudaEventRecord(d->ev[1], xs) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (launch_split_cols_s8(B, n, k, n, bp, stream) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (cudaStreamWaitEvent(stream, d->ev[1], 0) != cudaSuccess) return OZEMU_ERR_CUDA;
  return limb_gemm_s32(m, n, k, ap, bp, C32, n, d, stream);
}

size_t ozemu_four_plane_bytes(int rows, int k) {
  if (rows < 0 || k < 0) return 0;
  return four_plane_bytes(rows, k);
}

int ozemu_split_rows_s4(int rows, int k, const int8_t* X, int ldx, uint8_t* planes, cudaStream_t stream) {
  if (rows < 0 || k < 0 || ldx < (k > 1 ? k : 1)) return OZEMU_ERR_INVALID_ARG;
  if (rows == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !aligned16(planes) || !rows_ok(rows, 2)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (!four_tables().ok) return OZEMU_ERR_UNSUPPORTED;
  return cuda_status(launch_split_rows_four(X, ldx, rows, k, four_tables().a, planes, d->flags, stream));
}

int ozemu_split_cols_s8_four(int k, int cols, const int8_t* X, int ldx, uint8_t* planes, cudaStream_t stream) {
  if (k < 0 || cols < 0 || ldx < (cols > 1 ? cols : 1)) return OZEMU_ERR_INVALID_ARG;
  if (cols == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !aligned16(planes) || !rows_ok(cols, 2)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (!four_tables().ok) return OZEMU_ERR_UNSUPPORTED;
  if (k == 0) return OZEMU_OK;
  return cuda_status(launch_split_cols_four(X, ldx, k, cols, four_tables().b, planes, d->flags, stream));
}

int ozemu_igemm_s4s8(int m, int n, int k, const int8_t* A, const int8_t* B, int32_t* C32, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0) return OZEMU_ERR_INVALID_ARG;
  if (k > kMaxKS4) return OZEMU_ERR_K_OVERFLOW;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C32 || (k > 0 && (!A || !B)) || !rows_ok(m, 2) || !rows_ok(n, 2)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(launch_zero_s32(C32, m, n, n, stream));
  if (!four_tables().ok) return OZEMU_ERR_UNSUPPORTED;
  const size_t pa = align256(four_plane_bytes(m, k)), pb = align256(four_plane_bytes(n, k));
  uint8_t* ws = nullptr;
  s = workspace(d, pa + pb, &ws);
  if (s != OZEMU_OK) return s;
  uint8_t* ap = ws;
  uint8_t* bp = ws + pa;
  if (launch_split_rows_four(A, k, m, k, four_tables().a, ap, d->flags, stream) != cudaSuccess ||
      launch_split_cols_four(B, n, k, n, four_tables().b, bp, d->flags, stream) != cudaSuccess)
    return OZEMU_ERR_CUDA;
  LimbGemmCall c;
  c.residue_mode = false;
  c.m = m;
  c.n = n;
  c.k = k;
  c.r = 1;
  c.a_planes = ap;
  c.b_planes = bp;
  c.res_out = nullptr;
  c.ldr = 0;
  c.c32 = C32;
  c.ldc = n;
  c.kc_blocks = 64;  // exact chunks of 8192: |running sum| <= 1024 per K element
  c.limbs = 4;
  c.em = epi_moduli(1);
  c.flags = d->flags;
  return cuda_status(launch_limb_gemm(c, stream));
}

int ozemu_dgemm(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                int r, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || r < 1 || r > kMaxModuli) return OZEMU_ERR_INVALID_ARG;
  if (lda < (k > 1 ? k : 1) || ldb < (n > 1 ? n : 1) || ldc < (n > 1 ? n : 1)) return OZEMU_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C || (k > 0 && (!A || !B)) || !rows_ok(m, r) || !rows_ok(n, r)) return OZEMU_ERR_INVALID_ARG;
  int pa_bits = 0, pb_bits = 0;
  if (k > 0 && ozemu_bit_budget(k, r, &pa_bits, &pb_bits) != OZEMU_OK) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(launch_zero_f64(C, m, n, ldc, stream));
  if (n <= kNarrowMaxN && k <= kNarrowMaxK && pa_bits <= kNarrowMaxP && narrow_enabled())
    return dgemm_narrow(m, n, k, A, lda, B, ldb, C, ldc, r, pa_bits, pb_bits, d, stream);
  if (m >= 2048) return dgemm_chunked(m, n, k, A, lda, B, ldb, C, ldc, r, pa_bits, pb_bits, false, d, stream);
  const size_t pa = align256(plane_bytes(m, k, r)), pb = align256(plane_bytes(n, k, r));
  const size_t sa = align256(static_cast<size_t>(m) * 4), sb = align256(static_cast<size_t>(n) * 4);
  const size_t rb = align256(ozemu_residue_bytes(m, n, r));
  const size_t bt = colmax_bytes(n);  // column maxima of B
  uint8_t* ws = nullptr;
  s = workspace(d, pa + pb + sa + sb + rb + bt, &ws);
  if (s != OZEMU_OK) return s;
  uint8_t* ap = ws;
  uint8_t* bp = ap + pa;
  int32_t* sap = reinterpret_cast<int32_t*>(bp + pb);
  int32_t* sbp = reinterpret_cast<int32_t*>(bp + pb + sa);
  uint8_t* res = bp + pb + sa + sb;
  void* btr = res + rb;
  s = split_rows_f64(m, k, A, lda, pa_bits, r, ap, sap, d, stream);
  if (s != OZEMU_OK) return s;
  s = split_cols_f64(k, n, B, ldb, pb_bits, r, bp, sbp, btr, d, stream);
  if (s != OZEMU_OK) return s;
  s = residue_gemm(m, n, k, r, ap, bp, res, d, stream);
  if (s != OZEMU_OK) return s;
  return cuda_status(launch_crt_f64(m, n, res, round_up(n, 16), sap, sbp, C, ldc, crt_moduli(r), stream));
}

// ------------------------------------------- two-limb and mixed-digit moduli
// The entry points of the two families share these bodies; `limbs` names
// the list (2: two-limb, 1: mixed-digit).
static int family_moduli(int r, int32_t* out, int limbs) {
  if (r < 1 || r > max_r(limbs) || !out) return OZEMU_ERR_INVALID_ARG;
  for (int l = 0; l < r; ++l) out[l] = static_cast<int32_t>(moduli(limbs).m[l]);
  return OZEMU_OK;
}

static int family_bit_budget(int k, int r, int* p_a, int* p_b, int limbs) {
  if (k < 1 || r < 1 || r > max_r(limbs) || !p_a || !p_b) return OZEMU_ERR_INVALID_ARG;
  const int P = budget_P(k, r, limbs);
  if (P < 0) return OZEMU_ERR_INVALID_ARG;
  *p_a = (P + 1) / 2;
  *p_b = P / 2;
  return OZEMU_OK;
}

static size_t family_plane_bytes(int rows, int k, int r, int limbs) {
  if (rows < 0 || k < 0 || r < 1 || r > max_r(limbs)) return 0;
  return plane_bytes(rows, k, r, limbs);
}

static int family_split_rows(int rows, int k, const double* X, int ldx, int p, int r, uint8_t* planes,
                             int32_t* shifts, cudaStream_t stream, int limbs) {
  if (rows < 0 || k < 0 || ldx < (k > 1 ? k : 1) || p < 0 || p > 62 || r < 1 || r > max_r(limbs))
    return OZEMU_ERR_INVALID_ARG;
  if (rows == 0) return OZEMU_OK;
  if ((k > 0 && !X) || !planes || !shifts || !aligned16(planes) || !rows_ok(rows, r)) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  return split_rows_f64(rows, k, X, ldx, p, r, planes, shifts, d, stream, limbs);
}

static int family_dgemm(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                        int r, cudaStream_t stream, int limbs, bool from_host) {
  if (m < 0 || n < 0 || k < 0 || r < 1 || r > max_r(limbs)) return OZEMU_ERR_INVALID_ARG;
  if (lda < (k > 1 ? k : 1) || ldb < (n > 1 ? n : 1) || ldc < (n > 1 ? n : 1)) return OZEMU_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C || (k > 0 && (!A || !B)) || !rows_ok(m, r) || !rows_ok(n, r)) return OZEMU_ERR_INVALID_ARG;
  int pa_bits = 0, pb_bits = 0;
  if (k > 0 && family_bit_budget(k, r, &pa_bits, &pb_bits, limbs) != OZEMU_OK) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (from_host) {
    s = pipeline_state(d);
    if (s != OZEMU_OK) return s;
    if (k == 0) {
      uint8_t* buf = nullptr;
      s = workspace(d, align256(static_cast<size_t>(m) * n * 8), &buf);
      if (s != OZEMU_OK) return s;
      double* Cd = reinterpret_cast<double*>(buf);
      if (launch_zero_f64(Cd, m, n, n, stream) != cudaSuccess) return OZEMU_ERR_CUDA;
      return cuda_status(cudaMemcpy2DAsync(C, static_cast<size_t>(ldc) * 8, Cd, n * 8, static_cast<size_t>(n) * 8,
                                           m, cudaMemcpyDeviceToHost, stream));
    }
    return dgemm_chunked(m, n, k, A, lda, B, ldb, C, ldc, r, pa_bits, pb_bits, true, d, stream, limbs);
  }
  if (k == 0) return cuda_status(launch_zero_f64(C, m, n, ldc, stream));
  if (m >= 2048) return dgemm_chunked(m, n, k, A, lda, B, ldb, C, ldc, r, pa_bits, pb_bits, false, d, stream, limbs);
  const size_t pa = align256(plane_bytes(m, k, r, limbs)), pb = align256(plane_bytes(n, k, r, limbs));
  const size_t sa = align256(static_cast<size_t>(m) * 4), sb = align256(static_cast<size_t>(n) * 4);
  const size_t rb = align256(ozemu_residue_bytes(m, n, r));
  const size_t bt = colmax_bytes(n);  // column maxima of B
  uint8_t* ws = nullptr;
  s = workspace(d, pa + pb + sa + sb + rb + bt, &ws);
  if (s != OZEMU_OK) return s;
  uint8_t* ap = ws;
  uint8_t* bp = ap + pa;
  int32_t* sap = reinterpret_cast<int32_t*>(bp + pb);
  int32_t* sbp = reinterpret_cast<int32_t*>(bp + pb + sa);
  uint8_t* res = bp + pb + sa + sb;
  void* btr = res + rb;
  s = split_rows_f64(m, k, A, lda, pa_bits, r, ap, sap, d, stream, limbs);
  if (s != OZEMU_OK) return s;
  s = split_cols_f64(k, n, B, ldb, pb_bits, r, bp, sbp, btr, d, stream, limbs);
  if (s != OZEMU_OK) return s;
  s = residue_gemm(m, n, k, r, ap, bp, res, d, stream, limbs);
  if (s != OZEMU_OK) return s;
  return cuda_status(launch_crt_f64(m, n, res, round_up(n, 16), sap, sbp, C, ldc, crt_moduli(r, limbs), stream));
}

int ozemu_moduli_2limb(int r, int32_t* out) { return family_moduli(r, out, 2); }

int ozemu_bit_budget_2limb(int k, int r, int* p_a, int* p_b) { return family_bit_budget(k, r, p_a, p_b, 2); }

size_t ozemu_plane_bytes_2limb(int rows, int k, int r) { return family_plane_bytes(rows, k, r, 2); }

int ozemu_split_rows_f64_2limb(int rows, int k, const double* X, int ldx, int p, int r, uint8_t* planes,
                               int32_t* shifts, cudaStream_t stream) {
  return family_split_rows(rows, k, X, ldx, p, r, planes, shifts, stream, 2);
}

int ozemu_split_cols_f64_2limb(int k, int cols, const double* X, int ldx, int p, int r, uint8_t* planes,
                               int32_t* shifts, cudaStream_t stream) {
  return split_cols_entry(k, cols, X, ldx, p, r, planes, shifts, stream, 2);
}

int ozemu_residue_gemm_2limb(int m, int n, int k, int r, const uint8_t* a_planes, const uint8_t* b_planes,
                             uint8_t* residues, cudaStream_t stream) {
  return residue_gemm_entry(m, n, k, r, a_planes, b_planes, residues, stream, 2);
}

int ozemu_crt_f64_2limb(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a,
                        const int32_t* shifts_b, double* C, int ldc, cudaStream_t stream) {
  return crt_entry(m, n, r, residues, shifts_a, shifts_b, C, ldc, stream, 2);
}

int ozemu_dgemm_host_2limb(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C,
                           int ldc, int r, cudaStream_t stream) {
  return family_dgemm(m, n, k, A, lda, B, ldb, C, ldc, r, stream, 2, true);
}

int ozemu_dgemm_2limb(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                      int r, cudaStream_t stream) {
  return family_dgemm(m, n, k, A, lda, B, ldb, C, ldc, r, stream, 2, false);
}

int ozemu_max_moduli_mixed(void) { return kMaxModuliMix; }

int ozemu_single_digit_moduli_mixed(void) { return kMixSingle; }

int ozemu_moduli_mixed(int r, int32_t* out) { return family_moduli(r, out, 1); }

int ozemu_bit_budget_mixed(int k, int r, int* p_a, int* p_b) { return family_bit_budget(k, r, p_a, p_b, 1); }

size_t ozemu_plane_bytes_mixed(int rows, int k, int r) { return family_plane_bytes(rows, k, r, 1); }

int ozemu_products_mixed(int r) {
  if (r < 1 || r > kMaxModuliMix) return OZEMU_ERR_INVALID_ARG;
  const int single = single_count(r, 1);
  return single + 4 * (r - single);
}

int ozemu_split_rows_f64_mixed(int rows, int k, const double* X, int ldx, int p, int r, uint8_t* planes,
                               int32_t* shifts, cudaStream_t stream) {
  return family_split_rows(rows, k, X, ldx, p, r, planes, shifts, stream, 1);
}

int ozemu_split_cols_f64_mixed(int k, int cols, const double* X, int ldx, int p, int r, uint8_t* planes,
                               int32_t* shifts, cudaStream_t stream) {
  return split_cols_entry(k, cols, X, ldx, p, r, planes, shifts, stream, 1);
}

int ozemu_residue_gemm_mixed(int m, int n, int k, int r, const uint8_t* a_planes, const uint8_t* b_planes,
                             uint8_t* residues, cudaStream_t stream) {
  return residue_gemm_entry(m, n, k, r, a_planes, b_planes, residues, stream, 1);
}

int ozemu_crt_f64_mixed(int m, int n, int r, const uint8_t* residues, const int32_t* shifts_a,
                        const int32_t* shifts_b, double* C, int ldc, cudaStream_t stream) {
  return crt_entry(m, n, r, residues, shifts_a, shifts_b, C, ldc, stream, 1);
}

int ozemu_dgemm_mixed(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                      int r, cudaStream_t stream) {
  return family_dgemm(m, n, k, A, lda, B, ldb, C, ldc, r, stream, 1, false);
}

int ozemu_dgemm_host_mixed(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C,
                           int ldc, int r, cudaStream_t stream) {
  return family_dgemm(m, n, k, A, lda, B, ldb, C, ldc, r, stream, 1, true);
}

int ozemu_dgemm_host(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                     int r, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || r < 1 || r > kMaxModuli) return OZEMU_ERR_INVALID_ARG;
  if (lda < (k > 1 ? k : 1) || ldb < (n > 1 ? n : 1) || ldc < (n > 1 ? n : 1)) return OZEMU_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C || (k > 0 && (!A || !B)) || !rows_ok(m, r) || !rows_ok(n, r)) return OZEMU_ERR_INVALID_ARG;
  int pa_bits = 0, pb_bits = 0;
  if (k > 0 && ozemu_bit_budget(k, r, &pa_bits, &pb_bits) != OZEMU_OK) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  s = pipeline_state(d);
  if (s != OZEMU_OK) return s;
  const size_t szA = align256(static_cast<size_t>(m) * (k > 0 ? k : 1) * 8);
  const size_t szB = align256(static_cast<size_t>(k > 0 ? k : 1) * n * 8);
  const size_t szC = align256(static_cast<size_t>(m) * n * 8);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  const bool narrow = k == 0 || (n <= kNarrowMaxN && k <= kNarrowMaxK && pa_bits <= kNarrowMaxP && narrow_enabled());
  if (narrow) {
    // Small work: copy in, the device product, copy out, all on the caller's stream.
    uint8_t* buf = nullptr;
    s = workspace(d, szA + szB + szC + align256(static_cast<size_t>(n) * r * round_up(k > 0 ? k : 1, 16)) +
                         align256(static_cast<size_t>(n) * r * 4) + align256(ozemu_residue_bytes(m, n, r)) +
                         align256(static_cast<size_t>(m) * 4) + align256(static_cast<size_t>(n) * 4), &buf);
    if (s != OZEMU_OK) return s;
    double* Ad = reinterpret_cast<double*>(buf);
    double* Bd = reinterpret_cast<double*>(buf + szA);
    double* Cd = reinterpret_cast<double*>(buf + szA + szB);
    if (k == 0) {
      if (launch_zero_f64(Cd, m, n, n, stream) != cudaSuccess) return OZEMU_ERR_CUDA;
    } else {
      if (cudaMemcpy2DAsync(Ad, k * 8, A, static_cast<size_t>(lda) * 8, static_cast<size_t>(k) * 8, m, h2d, stream) !=
              cudaSuccess ||
          cudaMemcpy2DAsync(Bd, n * 8, B, static_cast<size_t>(ldb) * 8, static_cast<size_t>(n) * 8, k, h2d, stream) !=
              cudaSuccess)
        return OZEMU_ERR_CUDA;
      // The narrow path's own buffers follow the copies in the same workspace.
      uint8_t* rest = buf + szA + szB + szC;
      const size_t bres = align256(static_cast<size_t>(n) * r * round_up(k, 16));
      const size_t cs = align256(static_cast<size_t>(n) * r * 4);
      const size_t rb = align256(ozemu_residue_bytes(m, n, r));
      uint8_t* res = rest + bres + cs;
      int32_t* sap = reinterpret_cast<int32_t*>(res + rb);
      int32_t* sbp = reinterpret_cast<int32_t*>(res + rb + align256(static_cast<size_t>(m) * 4));
      NarrowCall c;
      c.m = m;
      c.n = n;
      c.k = k;
      c.kp = round_up(k, 16);
      c.pA = pa_bits;
      c.pB = pb_bits;
      c.A = Ad;
      c.lda = k;
      c.B = Bd;
      c.ldb = n;
      c.nm = narrow_moduli(r, pa_bits);
      c.ldr = round_up(n, 16);
      c.bres = rest;
      c.colsum = reinterpret_cast<int32_t*>(rest + bres);
      c.res = res;
      c.sa = sap;
      c.sb = sbp;
      c.flags = d->flags;
      if (launch_narrow_residues(c, stream) != cudaSuccess) return OZEMU_ERR_CUDA;
      if (launch_crt_f64(m, n, res, c.ldr, sap, sbp, Cd, n, crt_moduli(r), stream) != cudaSuccess)
        return OZEMU_ERR_CUDA;
    }
    return cuda_status(
        cudaMemcpy2DAsync(C, static_cast<size_t>(ldc) * 8, Cd, n * 8, static_cast<size_t>(n) * 8, m, d2h, stream));
  }

  return dgemm_chunked(m, n, k, A, lda, B, ldb, C, ldc, r, pa_bits, pb_bits, true, d, stream);
}

int ozemu_get_status(cudaStream_t stream) {
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return OZEMU_ERR_CUDA;
  uint32_t f = 0;
  if (cudaMemcpy(&f, d->flags, sizeof(f), cudaMemcpyDeviceToHost) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (cudaMemset(d->flags, 0, sizeof(f)) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (f & kFlagTimeout) return OZEMU_ERR_TIMEOUT;
  if (f & kFlagNonFinite) return OZEMU_ERR_NONFINITE;
  if (f & kFlagRange) return OZEMU_ERR_RANGE;
  return OZEMU_OK;
}

int ozemu_dgemm_noalloc(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C,
                        int ldc, int r, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0 || r < 1 || r > kMaxModuli) return OZEMU_ERR_INVALID_ARG;
  if (lda < (k > 1 ? k : 1) || ldb < (n > 1 ? n : 1) || ldc < (n > 1 ? n : 1)) return OZEMU_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OZEMU_OK;
  if (!C || (k > 0 && (!A || !B)) || !rows_ok(m, r) || !rows_ok(n, r)) return OZEMU_ERR_INVALID_ARG;
  int pa_bits = 0, pb_bits = 0;
  if (k > 0 && ozemu_bit_budget(k, r, &pa_bits, &pb_bits) != OZEMU_OK) return OZEMU_ERR_INVALID_ARG;
  const size_t fl = 256;
  const size_t pa = align256(plane_bytes(m, k, r)), pb = align256(plane_bytes(n, k, r));
  const size_t sa = align256(static_cast<size_t>(m) * 4), sb = align256(static_cast<size_t>(n) * 4);
  const size_t rb = align256(ozemu_residue_bytes(m, n, r));
  const size_t bt = colmax_bytes(n);  // column maxima of B
  if (k > 0 && fl + pa + pb + sa + sb + rb + bt > kNoAllocBytes) return OZEMU_ERR_SCRATCH_TOO_SMALL;
  uint8_t* base = nullptr;
  int s = noalloc_scratch(&base);
  if (s != OZEMU_OK) return s;
  if (k == 0) return cuda_status(launch_zero_f64(C, m, n, ldc, stream));
  // Only the status word must start at zero; every other part is fully
  // overwritten by the stage that produces it.
  if (cudaMemsetAsync(base, 0, fl, stream) != cudaSuccess) return OZEMU_ERR_CUDA;
  DeviceState d;
  d.flags = reinterpret_cast<uint32_t*>(base);
  uint8_t* ap = base + fl;
  uint8_t* bp = ap + pa;
  int32_t* sap = reinterpret_cast<int32_t*>(bp + pb);
  int32_t* sbp = reinterpret_cast<int32_t*>(bp + pb + sa);
  uint8_t* res = bp + pb + sa + sb;
  void* btr = res + rb;
  s = split_rows_f64(m, k, A, lda, pa_bits, r, ap, sap, &d, stream);
  if (s != OZEMU_OK) return s;
  s = split_cols_f64(k, n, B, ldb, pb_bits, r, bp, sbp, btr, &d, stream);
  if (s != OZEMU_OK) return s;
  s = residue_gemm(m, n, k, r, ap, bp, res, &d, stream);
  if (s != OZEMU_OK) return s;
  return cuda_status(launch_crt_f64(m, n, res, round_up(n, 16), sap, sbp, C, ldc, crt_moduli(r), stream));
}

int ozemu_get_status_noalloc(cudaStream_t stream) {
  uint8_t* base = nullptr;
  int s = noalloc_scratch(&base);
  if (s != OZEMU_OK) return s;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return OZEMU_ERR_CUDA;
  uint32_t f = 0;
  // A copy into a host variable and a fill of the word: nothing is allocated.
  if (cudaMemcpy(&f, base, sizeof(f), cudaMemcpyDeviceToHost) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (cudaMemset(base, 0, sizeof(f)) != cudaSuccess) return OZEMU_ERR_CUDA;
  if (f & kFlagTimeout) return OZEMU_ERR_TIMEOUT;
  if (f & kFlagNonFinite) return OZEMU_ERR_NONFINITE;
  return OZEMU_OK;
}

int ozemu_set_workspace_limit(size_t bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  std::lock_guard<std::mutex> lk(g_mu);
  g_ws_limit = bytes;
  if (bytes == 0 || dev < 0 || dev >= kMaxDevices) return OZEMU_OK;
  DeviceState& d = g_dev[dev];
  if (d.ws && d.ws_bytes > bytes) {  // the cached block is above the new cap: give it back
    cudaDeviceSynchronize();
    cudaFree(d.ws);
    d.ws = nullptr;
    d.ws_bytes = 0;
  }
  return OZEMU_OK;
}

size_t ozemu_workspace_limit(void) { return g_ws_limit; }

int ozemu_probe_wait_timeout(unsigned long long limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return OZEMU_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  int s = device_state(&d);
  if (s != OZEMU_OK) return s;
  wait_probe_kernel<<<1, 32, 0, stream>>>(d->flags, limit_ns);
  return cuda_status(cudaGetLastError());
}

void ozemu_release(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (d.ws) {
    cudaDeviceSynchronize();
    cudaFree(d.ws);
    d.ws = nullptr;
    d.ws_bytes = 0;
  }
}

}  // extern "C"
