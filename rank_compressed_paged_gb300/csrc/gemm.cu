// Tensor-core projections: the append's key / value projections (with, in the same
// launch, the decode's rank-space queries) and the chunked prefill's rank-space queries,
// as tcgen05 GEMMs D[128 x NT] = A[128 x K] * B[NT x K]^T.
//
// Both operands come from global memory through 2-D tensor maps with 128-byte swizzle
// (64 fp16 of K per row), four pipeline stages, one elected thread issuing
// tcgen05.mma.cta_group::1.kind::f16 into a TMEM accumulator.  When the token / query
// count is small, K is split over a thread-block cluster of KS CTAs; each CTA sends the
// rows owned by every peer to that peer's shared memory (distributed shared memory
// stores), a cluster barrier publishes them, and each CTA sums and writes its rows.
//
//   append, value job:  A = W_v rows [m0, m0+128) (K-major over H*d), B = v tokens,
//                       D[r][t] -> V page [slot_t / 16][slot_t % 16][m0 + r]
//   append, key job:    two heads h, h+1 at once as a block-diagonal product (K = 2d):
//                       A = [U_k,h 0; 0 U_k,h+1] (64-row boxes; the zero quadrants are
//                       boxes past the end of U_k, which the copy fills with zeros),
//                       B = k tokens of heads h and h+1 (adjacent columns),
//                       D[64 i + k][t] -> K page [slot_t / 16][h + i][slot_t % 16][k]
//   decode query job:   a key job with the decode queries as B (same launch as the
//                       append): D[64 i + k][q] = q~_{q,h+i,k}, stored fp32, scaled by
//                       log2(e)/sqrt(d), for the split-K scoring; a chunked prefill step
//                       puts its query projections (below) in the append's launch the
//                       same way.
//   query projection:   as a key job with the chunk's queries as B: D[k][q] = q~_{q,h,k},
//                       scaled by log2(e)/sqrt(d) and stored as an fp16 (hi, lo) pair
//                       (zero past r_k, up to 64), the prefill score MMA's A operand.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "rcp.h"
#include "shape.h"

namespace rcp {

constexpr int kGemmThreads = 128;
constexpr int kABytes = 128 * 64 * 2;   // one A stage: 128 rows x 64 K (or 64 K x 128 M)

enum GemmMode : int { kModeAppend = 0, kModeQproj = 2 };

template <int NT, int KS, int NB, int STG>
struct GemmSmem {
  static constexpr int B_BYTES = NT * 128;                     // one B operand stage
  static constexpr int STAGE = kABytes + NB * B_BYTES;
  // split-K receive buffer: KS partial slices of 128 / KS rows, rows RS floats apart (the
  // padding spreads the rows of a column over the banks)
  static constexpr int RS = NT + 4;
  static constexpr int RECV_OFF = STG * STAGE;
  static constexpr int RECV_BYTES = KS > 1 ? 128 * RS * 4 : 0;
  static constexpr int BAR_OFF = RECV_OFF + RECV_BYTES;        // full[S], empty[S], acc
  static constexpr int MISC_OFF = BAR_OFF + (2 * STG + 1) * 8;
  static constexpr int DST_OFF = MISC_OFF + 16;                // append: page offset per column
  static constexpr int RED_OFF = DST_OFF + NT * 8;             // 4-bit append: [4 warps][16]
  static constexpr int TOTAL = RED_OFF + 4 * 16 * 4;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr int TMEM_COLS = NT < 32 ? 32 : NT;
  static_assert(STAGE % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(MISC_OFF % 8 == 0 && DST_OFF % 8 == 0 && (RS * 4) % 16 == 0, "alignment");
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

struct GemmParams {
  // append
  const int64_t* slots;
  void* k_pages;
  void* v_pages;
  int32_t T;
  int32_t fmt;            // RCP_PAGES_*: fp16, E4M3 (round to nearest even, saturate) or
                          // 4-bit codes with per-group fp16 scales
  int64_t num_blocks;
  int32_t nq;             // decode queries (decode query jobs), prefill rows
  uint32_t* dev_err;
  // rank-space queries: chunked prefill fp16 hi / lo [nq][H][64]; decode fp32 [nq][H][r_k]
  void* qhi;
  void* qlo;
  float* qt;
  float qscale;
  int32_t wait_at_exit;   // wait for the previous launch at exit (one CTA) instead of first
};

// Where one CTA's job reads and writes.
struct GemmJob {
  int kind;        // 0 value (append), 1 key (append), 3 prefill query, 4 decode query,
                   // -1 idle
  int a_x, a_y;    // tensor-map coordinates of A's first k-block (x innermost)
  int b_x, b_y;    // coordinates of B's first k-block
  int a_step_x, a_step_y, b_step_x;   // per-k-block coordinate steps
  int kb0, kb1;    // k-block range of this CTA
  int m0;          // first output row (value rank row) / head index
  int n0;          // first token / query of the tile
  bool reduce;     // cluster split-K reduction
};

template <class S, int MODE, int NT, int KS>
__device__ __forceinline__ GemmJob gemm_job(uint32_t rank, int T, bool prefill_q) {
  GemmJob j{};
  const int cluster = blockIdx.x / KS;
  if constexpr (MODE == kModeAppend) {
    constexpr int NM = (S::R + 127) / 128;
    constexpr int NP = S::H / 2;                 // head pairs
    constexpr int NKG = (NP + KS - 1) / KS;
    constexpr int KBV = S::H * S::D / 64;
    constexpr int KBK = S::D / 64;
    // the append's clusters come first (the value jobs of every token tile, then their key
    // jobs), then the query jobs (head pairs, per query tile): decode or prefill queries
    const int app_clusters = (T + NT - 1) / NT * (NM + NKG);
    if (cluster >= app_clusters) {
      const int qc = cluster - app_clusters;
      const int pr = (qc % NKG) * KS + static_cast<int>(rank);
      j.kind = pr < NP ? (prefill_q ? 3 : 4) : -1;
      j.m0 = 2 * pr;
      j.n0 = (qc / NKG) * NT;
      j.kb0 = 0;
      j.kb1 = 2 * KBK;
      j.a_x = 0; j.a_y = j.m0 * S::RK; j.a_step_x = 64; j.a_step_y = 0;
      j.b_x = j.m0 * S::D; j.b_y = j.n0; j.b_step_x = 64;
      j.reduce = false;
      return j;
    }
    // value jobs of every token tile first (K = H d: the long ones, so they all start in
    // the first wave), then the key jobs
    const int ntile = (T + NT - 1) / NT;
    const bool value_job = cluster < ntile * NM;
    const int tile = value_job ? cluster / NM : (cluster - ntile * NM) / NKG;
    const int sub = value_job ? cluster % NM : NM + (cluster - ntile * NM) % NKG;
    j.n0 = tile * NT;
    if (sub < NM) {
      j.kind = 0;
      j.m0 = sub * 128;
      j.kb0 = static_cast<int>(rank) * KBV / KS;
      j.kb1 = (static_cast<int>(rank) + 1) * KBV / KS;
      j.a_x = j.kb0 * 64; j.a_y = j.m0; j.a_step_x = 64; j.a_step_y = 0;
      j.b_x = j.kb0 * 64; j.b_y = j.n0; j.b_step_x = 64;
      j.reduce = KS > 1;
    } else {
      const int pr = (sub - NM) * KS + static_cast<int>(rank);
      j.kind = pr < NP ? 1 : -1;
      j.m0 = 2 * pr;                             // first head of the pair
      j.kb0 = 0;
      j.kb1 = 2 * KBK;
      j.a_x = 0; j.a_y = j.m0 * S::RK; j.a_step_x = 64; j.a_step_y = 0;
      j.b_x = j.m0 * S::D; j.b_y = j.n0; j.b_step_x = 64;
      j.reduce = false;
    }
  } else if constexpr (MODE == kModeQproj) {
    // two heads h, h+1 at once, block-diagonal over K = 2d as the append's key jobs
    const int pr = blockIdx.x % (S::H / 2);
    j.kind = 3;
    j.m0 = 2 * pr;
    j.n0 = (blockIdx.x / (S::H / 2)) * NT;
    j.kb0 = 0;
    j.kb1 = 2 * (S::D / 64);
    j.a_x = 0; j.a_y = j.m0 * S::RK; j.a_step_x = 64; j.a_step_y = 0;
    j.b_x = j.m0 * S::D; j.b_y = j.n0; j.b_step_x = 64;
    j.reduce = false;
  }
  return j;
}

// Page offset (in fp16 elements; 4-bit pages: the slot itself) that column col of an append
// job writes from, or -1 when the token is padding (slot < 0), past the token count, or has
// an out-of-range slot (which also raises the device error bit).  Computed once per column
// before the epilogue so that the store loop issues no dependent loads.
template <class S>
__device__ __forceinline__ int64_t append_dst(const GemmParams& p, const GemmJob& j, int col) {
  const int n = j.n0 + col;
  if ((j.kind != 0 && j.kind != 1) || n >= p.T) return -1;
  const int64_t s = p.slots[n];
  if (s < 0) return -1;
  if (s >= p.num_blocks * kBlockSize) {
    atomicOr(p.dev_err, RCP_DEVERR_BAD_SLOT);
    return -1;
  }
  if (p.fmt == RCP_PAGES_INT4) return s;
  const int64_t blk = s / kBlockSize, off = s % kBlockSize;
  return j.kind == 0 ? (blk * kBlockSize + off) * S::R
                     : ((blk * S::H + j.m0) * kBlockSize + off) * S::RK;
}

// Round x / s to the nearest integer, ties to even, exactly for the fp32 x and fp16 s an
// append meets: k = rint(x * inv), inv a reciprocal of s within a few 2^-22 (relative), is
// within one of that integer (|x / s| <= 7), and the residual x - k s, which an fma computes
// exactly here (k s has at most 15 significant bits and lies within s of x), decides: beyond
// s / 2 the neighbour on its side, at s / 2 the even one.  No division, so no branch: the
// columns of an epilogue block interleave.
__device__ __forceinline__ int rne_div(float x, float s, float inv) {
  const float k = rintf(x * inv);
  const float r = fmaf(-k, s, x);
  const float a2 = 2.f * fabsf(r);
  const int ki = static_cast<int>(k);
  if (a2 > s || (a2 == s && (ki & 1) != 0)) return ki + (r > 0.f ? 1 : -1);
  return ki;
}

// 4-bit pages: quantize NC finished columns c0 .. c0+NC-1 of an append job, held by every
// thread as v[] for its row (TMEM lane), and store codes and scales.  A group is 64 rows:
// a key row of one head (rows 0..63, 64..127 of a key-pair job; rows at or past r_k of a
// head are not coefficients) or 64 value coefficients (m0 + 0..63, m0 + 64..127).  Per
// group: the smallest fp16 scale with 7 * scale >= max |x|, codes x / scale rounded to
// nearest, ties to even, in [-7, 7]; two codes per byte, the even row in the low nibble.
// All kGemmThreads threads take part (block barriers).
template <class S, int NC>
__device__ __forceinline__ void int4_store_columns(const GemmParams& p, const GemmJob& j,
                                                   const int64_t* dst, float* red, int c0,
                                                   const float* v) {
  using P = Int4Page<S>;
  const int row = threadIdx.x, warp = row >> 5, lane = row & 31;
  const bool valid = j.kind == 1 ? (row & 63) < S::RK : j.m0 + row < S::R;
  float a[NC];
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    a[e] = valid ? fabsf(v[e]) : 0.f;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a[e] = fmaxf(a[e], __shfl_xor_sync(0xffffffffu, a[e], o));
  }
  if (lane == 0)
#pragma unroll
    for (int e = 0; e < NC; ++e) red[warp * 16 + e] = a[e];
  __syncthreads();
  // every column's scale and code first (independent chains), then the stores
  __half shs[NC];
  int codes[NC];
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    const float amax = fmaxf(red[warp * 16 + e], red[(warp ^ 1) * 16 + e]);
    // the smallest fp16 h with 7 h >= amax: amax * (1/7) is within 2^-23 (relative) of
    // amax / 7, so h is that product rounded down or one of the next two fp16 values (7 h is
    // exact in fp32, so each test is exact)
    __half sh = __float2half_rd(amax * (1.f / 7.f));
#pragma unroll
    for (int up = 0; up < 2; ++up)
      if (__half2float(sh) * 7.f < amax)
        sh = __ushort_as_half(static_cast<unsigned short>(__half_as_ushort(sh) + 1));
    shs[e] = sh;
    const float sf = __half2float(sh);
    codes[e] = (valid && sf > 0.f) ? max(-7, min(7, rne_div(v[e], sf, __fdividef(1.f, sf)))) : 0;
  }
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    const __half sh = shs[e];
    const int code = codes[e];
    const int hi = __shfl_down_sync(0xffffffffu, code, 1);   // the next row's code
    const int64_t s = dst[c0 + e];
    if (s < 0 || !valid) continue;
    const int64_t blk = s / kBlockSize, off = s % kBlockSize;
    uint8_t* page;
    int64_t cbyte, sidx;
    bool first;   // the group's first row stores its scale
    if (j.kind == 1) {
      const int hh = j.m0 + (row >> 6), rr = row & 63;
      page = static_cast<uint8_t*>(p.k_pages) + blk * P::KBYTES;
      cbyte = ((hh * kBlockSize + off) * S::RK + rr) / 2;
      sidx = hh * kBlockSize + off;
      first = rr == 0;
      if (first) reinterpret_cast<__half*>(page + P::KCODES)[sidx] = sh;
    } else {
      const int r = j.m0 + row;
      page = static_cast<uint8_t*>(p.v_pages) + blk * P::VBYTES;
      cbyte = (off * S::R + r) / 2;
      sidx = off * (S::R / 64) + r / 64;
      first = (r & 63) == 0;
      if (first) reinterpret_cast<__half*>(page + P::VCODES)[sidx] = sh;
    }
    if ((row & 1) == 0) page[cbyte] = static_cast<uint8_t>((code & 0xF) | ((hi & 0xF) << 4));
  }
  __syncthreads();   // red[] is reused by the next call
}

// Write one finished output element (row, column) of a job.
template <class S>
__device__ __forceinline__ void gemm_store(const GemmParams& p, const GemmJob& j,
                                           const int64_t* dst, int row, int col, float v) {
  const int n = j.n0 + col;
  if (j.kind == 4) {
    // decode query: rows 0..63 are head m0's ranks, rows 64..127 head m0 + 1's
    const int hh = row >> 6, rr = row & 63;
    if (rr < S::RK && n < p.nq)
      p.qt[(static_cast<size_t>(n) * S::H + j.m0 + hh) * S::RK + rr] = v * p.qscale;
    return;
  }
  if (j.kind == 3) {
    // rows 0..63 are head m0's ranks, rows 64..127 head m0 + 1's; rows past r_k hold the
    // next heads' products and are written as the zero padding up to 64
    const int hh = row >> 6, rr = row & 63;
    if (n >= p.nq) return;
    const size_t at = (static_cast<size_t>(n) * S::H + j.m0 + hh) * 64 + rr;
    float q = rr < S::RK ? v * p.qscale : 0.f;
    const __half hi = __float2half_rn(q);
    static_cast<__half*>(p.qhi)[at] = hi;
    static_cast<__half*>(p.qlo)[at] = __float2half_rn(q - __half2float(hi));
    return;
  }
  const int64_t d = dst[col];
  if (d < 0) return;
  int64_t at;
  void* pages;
  if (j.kind == 0) {
    const int r = j.m0 + row;
    if (r >= S::R) return;
    at = d + r;
    pages = p.v_pages;
  } else {
    // rows 0..63 belong to head m0, rows 64..127 to head m0 + 1 (next head in the page)
    const int hh = row >> 6, rr = row & 63;
    if (rr >= S::RK) return;
    at = d + hh * kBlockSize * S::RK + rr;
    pages = p.k_pages;
  }
  if (p.fmt == RCP_PAGES_FP8_E4M3)
    static_cast<__nv_fp8_storage_t*>(pages)[at] = __nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
  else
    static_cast<__half*>(pages)[at] = __float2half_rn(v);
}

// One warp's epilogue staging area: 16 columns x 32 rows of at most 4 bytes (fp32 decode
// queries; the prefill queries' fp16 hi and lo parts take two 1 KB planes).
constexpr int kEpiWarpBytes = 16 * 32 * 4;

// Write columns c0 .. c0+15 of a job's tile for rows 32 warp .. 32 warp + 31 (v[] holds this
// lane's row).  In every destination a column's rows are contiguous (a page row's value
// coefficients, a head's ranks), so the warp transposes the block through its staging area
// and writes each column's run of rows as 16-byte pieces rather than an element per lane.
// ES: bytes per element (4 decode queries, 2 fp16 pages and prefill queries, 1 E4M3 pages);
// PL: planes (2 for the prefill queries' hi and lo parts).  Both fixed at compile time, so
// that the piece loop unrolls with shifts and masks for its indexes.
template <class S, int ES, int PL>
__device__ __forceinline__ void gemm_store_block(const GemmParams& p, const GemmJob& j,
                                                 const int64_t* dst, uint8_t* stage, int warp,
                                                 int lane, int c0, const float (&v)[16]) {
  static_assert(S::R % 32 == 0 && S::RK % 16 == 0, "runs of whole 16-byte pieces");
  constexpr int NCH = 32 * ES / 16;    // 16-byte pieces of a column's 32 rows, per plane
  constexpr int PER = 16 * NCH;        // pieces of the block, per plane
  static_assert((PL * PER) % 32 == 0 && PL * 16 * 32 * ES <= kEpiWarpBytes, "staging");
  const int hh = warp >> 1;            // key / query jobs: head m0 + hh
  const int rr0 = (warp & 1) * 32;     // ... ranks rr0 .. rr0 + 31
  int nvalid;
  if constexpr (ES == 4) {             // decode queries, fp32
    nvalid = min(32, max(0, S::RK - rr0));
    float* s = reinterpret_cast<float*>(stage);
#pragma unroll
    for (int e = 0; e < 16; ++e) s[e * 32 + lane] = v[e] * p.qscale;
  } else if constexpr (PL == 2) {      // prefill queries, fp16 hi and lo
    // ranks past r_k hold the next heads' products and are written as zero padding
    nvalid = 32;
    __half* s = reinterpret_cast<__half*>(stage);
    const bool rank = rr0 + lane < S::RK;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float q = rank ? v[e] * p.qscale : 0.f;
      const __half hi = __float2half_rn(q);
      s[e * 32 + lane] = hi;
      s[512 + e * 32 + lane] = __float2half_rn(q - __half2float(hi));
    }
  } else {                             // append: value or key page coefficients
    nvalid = j.kind == 0 ? min(32, max(0, S::R - (j.m0 + warp * 32)))
                         : min(32, max(0, S::RK - rr0));
    if constexpr (ES == 1) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        stage[e * 32 + lane] = __nv_cvt_float_to_fp8(v[e], __NV_SATFINITE, __NV_E4M3);
    } else {
      __half* s = reinterpret_cast<__half*>(stage);
#pragma unroll
      for (int e = 0; e < 16; ++e) s[e * 32 + lane] = __float2half_rn(v[e]);
    }
  }
  __syncwarp();
  const int nvc = nvalid * ES / 16;    // pieces of a column that hold valid rows
#pragma unroll
  for (int it = 0; it < PL * PER / 32; ++it) {
    const int i = lane + 32 * it;
    const int plane = i / PER, c = (i % PER) / NCH, k = i % NCH;
    if (k >= nvc) continue;
    uint8_t* out;
    if constexpr (ES == 4 || PL == 2) {
      const int n = j.n0 + c0 + c;
      if (n >= p.nq) continue;
      const size_t hrow = static_cast<size_t>(n) * S::H + j.m0 + hh;
      if constexpr (ES == 4)
        out = reinterpret_cast<uint8_t*>(p.qt) + (hrow * S::RK + rr0) * 4;
      else
        out = static_cast<uint8_t*>(plane ? p.qlo : p.qhi) + (hrow * 64 + rr0) * 2;
    } else {
      const int64_t d = dst[c0 + c];
      if (d < 0) continue;
      out = j.kind == 0
                ? static_cast<uint8_t*>(p.v_pages) + (d + j.m0 + warp * 32) * ES
                : static_cast<uint8_t*>(p.k_pages) + (d + hh * kBlockSize * S::RK + rr0) * ES;
    }
    *reinterpret_cast<uint4*>(out + k * 16) =
        *reinterpret_cast<const uint4*>(stage + plane * 1024 + c * 32 * ES + k * 16);
  }
  __syncwarp();   // the staging area is rewritten by the next block
}

template <class S, int MODE, int NT, int KS, int STG>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a2,
                const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b2,
                const __grid_constant__ CUtensorMap map_b3, const GemmParams p) {
  constexpr int kGemmStages = STG;
  using L = GemmSmem<NT, KS, 1, STG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
  uint64_t* empty = full + kGemmStages;
  uint64_t* accb = empty + kGemmStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);
  float* recv = reinterpret_cast<float*>(sm + L::RECV_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = KS > 1 ? cluster_ctarank() : 0;
  const GemmJob j = gemm_job<S, MODE, NT, KS>(rank, p.T, p.qhi != nullptr);
  // value jobs read W_v through map_a and their tokens through map_b;
  // key jobs (and the query jobs of the query-projection launch) read U_k through map_a2
  // and their rows through map_b2; query jobs of an append launch read U_k through map_a2
  // and the queries through map_b3
  const bool uk = j.kind == 1 || j.kind == 3 || j.kind == 4;
  const bool qjob = j.kind == 4 || (MODE == kModeAppend && j.kind == 3);
  const CUtensorMap* amap = uk ? &map_a2 : &map_a;
  const CUtensorMap* bmap = qjob ? &map_b3 : (uk ? &map_b2 : &map_b);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemmStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (j.reduce) cluster_sync_all();   // every peer is running before any remote store

  const int nkb = j.kind >= 0 ? j.kb1 - j.kb0 : 0;
  auto load_a = [&](int kb, int s) {
    uint8_t* st = sm + s * L::STAGE;
    if ((MODE == kModeAppend && (j.kind == 1 || j.kind == 3 || j.kind == 4)) ||
        MODE == kModeQproj) {
      // block-diagonal pair: k-blocks [0, d/64) meet head m0's rows (top), the rest head
      // m0 + 1's (bottom); the other half is a box past the last row of U_k (zeros)
      constexpr int KBK = S::D / 64, OOB = S::H * S::RK;
      const int half = kb / KBK, kk = kb % KBK;
      tma_load_2d(st, amap, kk * 64, half == 0 ? j.m0 * S::RK : OOB, &full[s]);
      tma_load_2d(st + kABytes / 2, amap, kk * 64, half == 1 ? (j.m0 + 1) * S::RK : OOB, &full[s]);
    } else {
      tma_load_2d(st, amap, j.a_x + kb * j.a_step_x, j.a_y, &full[s]);
    }
  };
  auto load_b = [&](int kb, int s) {
    uint8_t* st = sm + s * L::STAGE;
    tma_load_2d(st + kABytes, bmap, j.b_x + kb * j.b_step_x, j.b_y, &full[s]);
  };
  // A is always a factor (W_v or U_k), which no kernel writes: its first stages are
  // fetched before waiting on the previous kernel, whose outputs only B may read.
  constexpr uint32_t kStageTx = kABytes + L::B_BYTES;
  const int pre = nkb < kGemmStages ? nkb : kGemmStages;
  if (warp == 0 && lane == 0 && nkb > 0) {
    prefetch_tmap(amap);
    prefetch_tmap(bmap);
    for (int kb = 0; kb < pre; ++kb) {
      mbar_arrive_expect_tx(&full[kb], kStageTx);
      load_a(kb, kb);
    }
  }
  // operands written by the previous kernel are visible (unless that kernel writes nothing
  // this one touches: then it is waited for at exit, so that kernels after this one still
  // see its results)
  if (!p.wait_at_exit) griddep_wait();
  griddep_launch();

  if (warp == 0 && lane == 0 && nkb > 0) {
    // -------------------------------------------------------------- TMA producer
    int issued = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % kGemmStages;
      if (kb >= pre) {
        if (!mbar_wait(&empty[s], ((kb / kGemmStages) - 1) & 1, abort_flag, p.dev_err)) break;
        mbar_arrive_expect_tx(&full[s], kStageTx);
        load_a(kb, s);
      }
      load_b(kb, s);
      ++issued;
    }
    if (*abort_flag)
      for (int i = (issued > kGemmStages ? issued - kGemmStages : 0); i < issued; ++i)
        mbar_wait_drain(&full[i % kGemmStages], (i / kGemmStages) & 1);
  } else if (warp == 1 && lane == 0 && nkb > 0) {
    // -------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = make_idesc_f16(128, NT, false, false);
    int kb = 0;
    for (; kb < nkb; ++kb) {
      const int s = kb % kGemmStages;
      if (!mbar_wait(&full[s], (kb / kGemmStages) & 1, abort_flag, p.dev_err)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sm + s * L::STAGE);
      const uint32_t b0 = a0 + kABytes;
#pragma unroll
      for (int k = 0; k < 4; ++k) {   // four K=16 steps per 64-wide k-block
        const uint64_t ad = make_sdesc(a0 + k * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = make_sdesc(b0 + k * 32, 16, 1024, kSwizzle128B);
        umma_f16(tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(accb);
    if (kb < nkb) mbar_wait_drain(accb, 0);
  }
  __syncwarp();
  int64_t* dst_s = reinterpret_cast<int64_t*>(sm + L::DST_OFF);
  if (MODE == kModeAppend) {
    // idle warps get here while the main loop runs; the two issuing lanes join after it
    for (int c = threadIdx.x; c < NT; c += kGemmThreads) dst_s[c] = append_dst<S>(p, j, c);
    __syncthreads();
  }

  // ------------------------------------------------------------------ epilogue
  // warp-uniform, since TMEM loads are warp-collective
  const bool have_acc = __all_sync(0xffffffffu, nkb > 0 && mbar_wait(accb, 0, abort_flag, p.dev_err));
  tc_fence_after();
  const int row = warp * 32 + lane;                          // TMEM lane = output row
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  // 4-bit pages: an append job quantizes whole 64-row groups (uniform over the CTA, and
  // over the cluster for split-K value jobs)
  const bool int4 = MODE == kModeAppend && p.fmt == RCP_PAGES_INT4 && (j.kind == 0 || j.kind == 1);
  float* red = reinterpret_cast<float*>(sm + L::RED_OFF);
  if (int4 && !j.reduce) {
#pragma unroll 1
    for (int c0 = 0; c0 < NT; c0 += 16) {
      float v[16];
      if (have_acc) {
        tmem_ld16(trow + c0, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.f;
      }
      int4_store_columns<S, 16>(p, j, dst_s, red, c0, v);
    }
  } else if (int4) {
    if constexpr (KS > 1) {
    // split-K: column c belongs to peer c / CPC, which receives every row of it (a group
    // spans 64 rows) in slot [my rank][row][c % CPC]
    constexpr int CPC = NT / KS;
    static_assert(CPC >= 1 && CPC <= 16 && NT % KS == 0, "4-bit split-K columns");
    const uint32_t recv_local = smem_u32(recv);
#pragma unroll 1
    for (int c0 = 0; c0 < NT; c0 += 16) {
      float v[16];
      if (have_acc) {
        tmem_ld16(trow + c0, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.f;
      }
      if constexpr (CPC % 4 == 0) {   // four columns of one peer per 16-byte store
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
          const int col = c0 + e;
          st_cluster_v4(map_to_rank(recv_local, static_cast<uint32_t>(col / CPC)) +
                            ((rank * 128 + row) * CPC + col % CPC) * 4,
                        v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int col = c0 + e;
          st_cluster_f32(map_to_rank(recv_local, static_cast<uint32_t>(col / CPC)) +
                             ((rank * 128 + row) * CPC + col % CPC) * 4,
                         v[e]);
        }
      }
    }
    cluster_sync_all();
    float v[CPC];
#pragma unroll
    for (int c = 0; c < CPC; ++c) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < KS; ++s) acc += recv[(s * 128 + row) * CPC + c];
      v[c] = acc;
    }
    int4_store_columns<S, CPC>(p, j, dst_s, red, static_cast<int>(rank) * CPC, v);
    }
  } else if (!j.reduce) {
    if (have_acc) {
      // the pipeline stages are idle once the accumulator is complete: each warp stages its
      // blocks in the first stage
      static_assert(4 * kEpiWarpBytes <= L::STAGE, "epilogue staging fits in one stage");
      uint8_t* stage = sm + warp * kEpiWarpBytes;
      auto blocks = [&](auto store) {
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 16) {
          float v[16];
          tmem_ld16(trow + c0, v);
          tmem_wait_ld();
          store(c0, v);
        }
      };
      if (j.kind == 4)
        blocks([&](int c0, const float(&v)[16]) { gemm_store_block<S, 4, 1>(p, j, dst_s, stage, warp, lane, c0, v); });
      else if (j.kind == 3)
        blocks([&](int c0, const float(&v)[16]) { gemm_store_block<S, 2, 2>(p, j, dst_s, stage, warp, lane, c0, v); });
      else if (p.fmt == RCP_PAGES_FP8_E4M3)
        blocks([&](int c0, const float(&v)[16]) { gemm_store_block<S, 1, 1>(p, j, dst_s, stage, warp, lane, c0, v); });
      else
        blocks([&](int c0, const float(&v)[16]) { gemm_store_block<S, 2, 1>(p, j, dst_s, stage, warp, lane, c0, v); });
    }
  } else {
    // split-K: row r belongs to peer r / RPC; send it to slot [my rank] of that peer
    constexpr int RPC = 128 / KS;
    const uint32_t recv_local = smem_u32(recv);
    const uint32_t dst_rank = static_cast<uint32_t>(row / RPC);
    const uint32_t dst = map_to_rank(recv_local, dst_rank) +
                         ((rank * RPC + (row % RPC)) * L::RS) * 4;
#pragma unroll 1
    for (int c0 = 0; c0 < NT; c0 += 16) {
      float v[16];
      if (have_acc) {
        tmem_ld16(trow + c0, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        st_cluster_v4(dst + (c0 + e) * 4, v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
    cluster_sync_all();
    // sum the KS partial slices of my RPC rows and write them
    for (int i = threadIdx.x; i < RPC * NT; i += kGemmThreads) {
      const int rr = i % RPC, col = i / RPC;
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < KS; ++s) acc += recv[(s * RPC + rr) * L::RS + col];
      gemm_store<S>(p, j, dst_s, static_cast<int>(rank) * RPC + rr, col, acc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
  // the launch before is waited for by one CTA: this grid cannot complete until that CTA
  // leaves, so kernels after it still find the earlier launch complete, while the short
  // jobs' CTAs leave their SMs at once (CTA 0 runs a value job, the longest)
  if (p.wait_at_exit && blockIdx.x == 0) griddep_wait();
}

// --------------------------------------------------------------------------- launchers
template <class K>
static cudaError_t launch_cluster(K kernel, int grid, int cluster, int smem, cudaStream_t stream,
                                  bool pdl, const CUtensorMap& a, const CUtensorMap& a2,
                                  const CUtensorMap& b, const CUtensorMap& b2,
                                  const CUtensorMap& b3, const GemmParams& p) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, a, a2, b, b2, b3, p);
}

// Append: small token counts split K over an 8-CTA cluster (64-token tiles); large ones
// use 256-token tiles without a split.
template <class S>
struct AppendCfg {
  static constexpr int KS_SMALL = (S::H * S::D / 64) < 8 ? (S::H * S::D / 64) : 8;
  // pipeline stages by token tile: every k-block of a split-K value job (or of a key /
  // query job) in flight at once where shared memory allows
  static constexpr int STG16 = 8, STG64 = 6, STG256 = 4;
};

template <class S>
cudaError_t prepare_gemm() {
  cudaError_t e;
  auto set = [&](auto kernel, int smem) {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    return r;
  };
  using AC = AppendCfg<S>;
  constexpr int KSS = AC::KS_SMALL;
  if ((e = set(gemm_kernel<S, kModeAppend, 16, KSS, AC::STG16>,
               GemmSmem<16, KSS, 1, AC::STG16>::ALLOC)) != cudaSuccess)
    return e;
  if ((e = set(gemm_kernel<S, kModeAppend, 64, KSS, AC::STG64>,
               GemmSmem<64, KSS, 1, AC::STG64>::ALLOC)) != cudaSuccess)
    return e;
  if ((e = set(gemm_kernel<S, kModeAppend, 256, 1, AC::STG256>,
               GemmSmem<256, 1, 1, AC::STG256>::ALLOC)) != cudaSuccess)
    return e;
  if ((e = set(gemm_kernel<S, kModeQproj, 64, 1, 2>, GemmSmem<64, 1, 1, 2>::ALLOC)) != cudaSuccess)
    return e;
  if ((e = set(gemm_kernel<S, kModeQproj, 256, 1, 2>, GemmSmem<256, 1, 1, 2>::ALLOC)) != cudaSuccess)
    return e;
  return cudaSuccess;
}

// The append's projections and, when ap.nq > 0, the rank-space queries (a decode's, or a
// chunked prefill step's when ap.qhi is set), in one launch (either part may be empty).  q_rows: tensor map over the queries [nq][H*d] with
// the same box as the token maps (64 x 64 when max(T, nq) <= 256, else 64 x 256).
template <class S>
cudaError_t launch_append_gemm(const CUtensorMap& w_v, const CUtensorMap& u_k,
                               const CUtensorMap& v_rows, const CUtensorMap& k_rows,
                               const CUtensorMap& q_rows, const AppendParams& ap,
                               cudaStream_t stream) {
  if (ap.T == 0 && ap.nq == 0) return cudaSuccess;
  GemmParams p{};
  p.slots = ap.slots;
  p.k_pages = ap.k_pages;
  p.v_pages = ap.v_pages;
  p.T = ap.T;
  p.fmt = ap.page_format;
  p.num_blocks = ap.num_blocks;
  p.dev_err = ap.dev_err;
  p.qt = ap.qt;
  p.qhi = ap.qhi;
  p.qlo = ap.qlo;
  p.nq = ap.nq;
  p.qscale = ap.qscale;
  p.wait_at_exit = ap.wait_at_exit;
  using AC = AppendCfg<S>;
  constexpr int NM = (S::R + 127) / 128;
  constexpr int KS = AC::KS_SMALL;
  constexpr int NKG = (S::H / 2 + KS - 1) / KS;
  const int rows = ap.T > ap.nq ? ap.T : ap.nq;
  if (rows <= 16) {   // a decode step of up to 16 requests: 16-row tiles
    const int clusters = (ap.T + 15) / 16 * (NM + NKG) + (ap.nq + 15) / 16 * NKG;
    return launch_cluster(gemm_kernel<S, kModeAppend, 16, KS, AC::STG16>, clusters * KS, KS,
                          GemmSmem<16, KS, 1, AC::STG16>::ALLOC, stream, true, w_v, u_k, v_rows,
                          k_rows, q_rows, p);
  }
  if (rows <= 256) {
    const int clusters = (ap.T + 63) / 64 * (NM + NKG) + (ap.nq + 63) / 64 * NKG;
    return launch_cluster(gemm_kernel<S, kModeAppend, 64, KS, AC::STG64>, clusters * KS, KS,
                          GemmSmem<64, KS, 1, AC::STG64>::ALLOC, stream, true, w_v, u_k, v_rows,
                          k_rows, q_rows, p);
  }
  // many tokens or queries: 256-row tiles, no split
  const int clusters = (ap.T + 255) / 256 * (NM + S::H / 2) + (ap.nq + 255) / 256 * (S::H / 2);
  return launch_cluster(gemm_kernel<S, kModeAppend, 256, 1, AC::STG256>, clusters, 1,
                        GemmSmem<256, 1, 1, AC::STG256>::ALLOC, stream, true, w_v, u_k, v_rows,
                        k_rows, q_rows, p);
}

template <class S>
cudaError_t launch_qproj_gemm(const CUtensorMap& u_k, const CUtensorMap& q_rows, void* qhi,
                              void* qlo, int nq, float qscale, uint32_t* dev_err,
                              cudaStream_t stream, bool pdl) {
  GemmParams p{};
  p.nq = nq;
  p.qhi = qhi;
  p.qlo = qlo;
  p.qscale = qscale;
  p.dev_err = dev_err;
  if (nq <= 256) {
    const int tiles = (nq + 63) / 64;
    return launch_cluster(gemm_kernel<S, kModeQproj, 64, 1, 2>, tiles * (S::H / 2), 1,
                          GemmSmem<64, 1, 1, 2>::ALLOC, stream, pdl, u_k, u_k, q_rows, q_rows,
                          q_rows, p);
  }
  const int tiles = (nq + 255) / 256;
  return launch_cluster(gemm_kernel<S, kModeQproj, 256, 1, 2>, tiles * (S::H / 2), 1,
                        GemmSmem<256, 1, 1, 2>::ALLOC, stream, pdl, u_k, u_k, q_rows, q_rows,
                        q_rows, p);
}

template cudaError_t prepare_gemm<ShapeMain>();
template cudaError_t prepare_gemm<ShapeTiny>();
template cudaError_t launch_append_gemm<ShapeMain>(const CUtensorMap&, const CUtensorMap&,
                                                   const CUtensorMap&, const CUtensorMap&,
                                                   const CUtensorMap&, const AppendParams&,
                                                   cudaStream_t);
template cudaError_t launch_append_gemm<ShapeTiny>(const CUtensorMap&, const CUtensorMap&,
                                                   const CUtensorMap&, const CUtensorMap&,
                                                   const CUtensorMap&, const AppendParams&,
                                                   cudaStream_t);
template cudaError_t launch_qproj_gemm<ShapeMain>(const CUtensorMap&, const CUtensorMap&, void*,
                                                  void*, int, float, uint32_t*, cudaStream_t,
                                                  bool);
template cudaError_t launch_qproj_gemm<ShapeTiny>(const CUtensorMap&, const CUtensorMap&, void*,
                                                  void*, int, float, uint32_t*, cudaStream_t,
                                                  bool);

}  // namespace rcp
