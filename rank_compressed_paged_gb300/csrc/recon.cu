// Value reconstruction for the reconstructing chunked prefill: V^ = C_v W_v for every
// cached key of the requests that have chunk rows, on tensor cores.
//
// The Proxima page's prefill kernel ("Per-prefill-chunk attention") expands compressed K
// from its low-rank basis per query tile.  Here the keys stay in rank space (r_k = 64 per
// head is cheaper than d = 128) and the joint value coefficients are expanded instead:
// with R = 1024 and d = 128 that costs R*H*d multiply-adds per key once, against R per
// (query row, key, head) in rank space, so it does less work once a chunk has more than
// R*d/(R-d) ~ 146 rows per request.
//
// The keys of all such requests, page after page in request order (prefix sums in
// vcum), are the rows of one GEMM D[keys x H*d] = C_v[keys x R] * W_v[R x H*d], cut into
// tiles of 256 keys (16 pages) x 256 columns:
//   * persistent CTA pairs (one CTA per SM) take the tiles in turn; each CTA stages its 128
//     keys' C_v rows (A: one 16 x 64 tensor-map box per page per 64-wide k-block, K-major,
//     128-byte swizzle) and half of the W_v tile (B: 128 columns, two 64 x 64 boxes,
//     MN-major), so a k-block costs each SM 32 KB of operands instead of the 48 KB of a
//     one-CTA 128 x 256 tile;
//   * a page holds only 16 keys, and the copy engine's cost per box set the kernel's pace
//     with eight C_v boxes per CTA per k-block; so (when the columns split into an even
//     number of tiles) two pairs form a 4-CTA cluster on one row of keys and adjacent
//     column tiles, and each CTA copies half of its eight C_v boxes, multicast to itself
//     and to the CTA holding the same keys in the other pair: six boxes per k-block;
//   * both CTAs' copies of a pair (multicast ones included) complete on the pair's even-CTA
//     stage barrier; the even CTA issues tcgen05.mma.cta_group::2, M=256, N=256, K=16
//     steps; each commit frees the stage in every CTA of the cluster (a stage is refilled
//     only when both pairs have read it); a CTA's tensor memory holds two 256-column
//     accumulators of its 128 rows, so the epilogue of one tile overlaps the MMAs of the
//     next;
//   * four epilogue warps write V^ rows as fp16, zero for the slots of a page past the end
//     of its sequence (so that the attention can never meet 0 * NaN there).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "rcp.h"
#include "shape.h"

namespace rcp {

// warp 0 copies, warp 1 issues the MMAs (even CTA), warps 2-5 the epilogue, warp 6 looks
// up the pages of the tiles ahead
constexpr int kRcThreads = 224;
constexpr int kRcRing = 4;   // tiles whose page rows are looked up ahead

template <class S>
struct ReconSmem {
  using C = ReconCfg<S>;
  static constexpr int A_BYTES = C::MT * 128;          // 128 keys x 64 ranks
  static constexpr int B_BYTES = C::NTC * 128;         // 64 ranks x 128 columns
  static constexpr int STAGE = A_BYTES + B_BYTES;
  // the epilogue warps' staging buffers: 32 rows x 64 columns of fp16 each (16-byte chunk c
  // of row r at chunk c ^ (r % 8)), so that V^ leaves in whole 128-byte row pieces
  static constexpr int EPI_OFF = C::STG * STAGE;
  static constexpr int EPI_BYTES = 32 * 128;
  // the page rows of the next tiles: [kRcRing][8] TMA row coordinates
  static constexpr int ROW_OFF = EPI_OFF + 4 * EPI_BYTES;
  // full[STG] (even CTA), empty[STG], tfull[2], tempty[2] (even CTA), rfull / rempty[kRcRing]
  static constexpr int BAR_OFF = ROW_OFF + kRcRing * 8 * 4;
  static constexpr int MISC_OFF = BAR_OFF + (2 * C::STG + 4 + 2 * kRcRing) * 8;   // tmem slot, abort
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr int TMEM_COLS = 2 * C::NT;          // two accumulators
  static_assert(STAGE % 1024 == 0, "stages keep 1024-byte alignment");
  // more than half an SM's shared memory: one CTA per SM, so the two CTAs of a pair always
  // sit on two SMs and each has the SM's whole tensor memory
  static_assert(2 * ALLOC > 228 * 1024 && ALLOC <= 227 * 1024, "one CTA per SM");
};

// CTA pairs per cluster: two when the column tiles pair up, else one
template <class S>
constexpr int recon_pairs() {
  return (S::H * S::D / ReconCfg<S>::NT) % 2 == 0 ? 2 : 1;
}

template <class S>
__global__ void __launch_bounds__(kRcThreads, 1)
    recon_kernel(const __grid_constant__ CUtensorMap vp_map, const __grid_constant__ CUtensorMap w_map,
                 const AttnParams p) {
  using C = ReconCfg<S>;
  using L = ReconSmem<S>;
  constexpr int HD = S::H * S::D, NTN = HD / C::NT, BPT = C::MT / kBlockSize;
  constexpr int P = recon_pairs<S>(), CL = 2 * P;   // pairs, CTAs per cluster
  constexpr int NU = NTN / P;                       // column units of a row tile
  constexpr int BPC = BPT / P;                      // C_v boxes a CTA issues per k-block
  static_assert(NTN % P == 0 && BPT % P == 0, "cluster split");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
  uint64_t* empty = full + C::STG;
  uint64_t* tfull = empty + C::STG;    // [2] accumulator b holds a finished tile
  uint64_t* tempty = tfull + 2;        // [2] ... and both CTAs' epilogues have read it
  uint64_t* rfull = tempty + 2;        // [kRcRing] a tile's page rows are written
  uint64_t* rempty = rfull + kRcRing;  // [kRcRing] ... and were read
  int32_t* rows_s = reinterpret_cast<int32_t*>(sm + L::ROW_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int h = static_cast<int>(rank & 1);          // half of the pair (0 issues the MMAs)
  const int pr = static_cast<int>(rank >> 1);        // pair of the cluster
  const uint32_t lead = rank & ~1u;                  // the pair's even CTA
  const int64_t cid = blockIdx.x / CL, ncl = gridDim.x / CL;   // cluster, clusters

  griddep_wait();   // page prefix sums (plan) and the appended chunk are visible
  griddep_launch();
  const int64_t total = p.vcum[p.batch];
  const int64_t ntiles = (total + 2 * BPT - 1) / (2 * BPT) * NU;   // cluster work units
  if (cid >= ntiles) return;   // uniform over the cluster, before any cluster operation
  // unit t: keys of pages [16 (t / NU), +16), pair pr's columns [256 ct, +256) with
  // ct = (t % NU) P + pr; this CTA's keys are pages 16 (t / NU) + 8 h .. + 8, of which it
  // copies the BPC starting at 8 h + BPC pr

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STG; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], P);   // a commit of every pair of the cluster
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * 4);   // the four epilogue warps of each CTA
    }
    for (int r = 0; r < kRcRing; ++r) {
      mbar_init(&rfull[r], 1);
      mbar_init(&rempty[r], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, L::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();   // every CTA's barriers exist before any copy or arrival reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto col_tile = [&](int64_t t) { return static_cast<int>(t % NU) * P + pr; };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ copies
    prefetch_tmap(&vp_map);
    prefetch_tmap(&w_map);
    constexpr uint16_t kMcast = P == 2 ? 0x5 : 0x1;   // same half of both pairs
    int64_t n = 0;   // k-blocks issued (stage n % STG)
    bool ok = true;
    for (int64_t t = cid, i = 0; ok && t < ntiles; t += ncl, ++i) {
      const int r = static_cast<int>(i % kRcRing);
      if (!mbar_wait(&rfull[r], (i / kRcRing) & 1, abort_flag, p.dev_err)) break;
      int32_t yrow[BPC];
#pragma unroll
      for (int jb = 0; jb < BPC; ++jb) yrow[jb] = rows_s[r * 8 + jb];
      mbar_arrive(&rempty[r]);
      const int x0 = col_tile(t) * C::NT + h * C::NTC;
      for (int kb = 0; kb < C::KB; ++kb, ++n) {
        const int s = static_cast<int>(n % C::STG);
        if (n >= C::STG &&
            !mbar_wait(&empty[s], ((n / C::STG) - 1) & 1, abort_flag, p.dev_err)) {
          ok = false;
          break;
        }
        uint8_t* st = sm + s * L::STAGE;
        const uint32_t fb = map_to_rank(smem_u32(&full[s]), lead);
        // the pair's A (from every issuer) and B, in both CTAs
        if (h == 0) mbar_arrive_expect_tx(&full[s], 2 * L::STAGE);
#pragma unroll
        for (int jb = 0; jb < BPC; ++jb) {
          uint8_t* dst = st + (pr * BPC + jb) * 2048;
          if constexpr (P == 2)
            tma_load_2d_mc_pair(dst, &vp_map, kb * 64, yrow[jb], fb, kMcast << h);
          else
            tma_load_2d_pair(dst, &vp_map, kb * 64, yrow[jb], fb);
        }
#pragma unroll
        for (int q = 0; q < C::NTC / 64; ++q)
          tma_load_2d_pair(st + L::A_BYTES + q * 8192, &w_map, x0 + q * 64, kb * 64, fb);
      }
    }
    // the commits of the last stages (arrivals on this CTA's barriers) land before it exits
    for (int64_t i = (n > C::STG ? n - C::STG : 0); i < n; ++i)
      mbar_wait_drain(&empty[i % C::STG], (i / C::STG) & 1);
  } else if (warp == 6) {
    // ------------------------------------------------------------------- page lookups
    // lane j < BPC resolves the j-th page this CTA copies of each unit (page BPC pr + j of
    // its half): its TMA row, or row -16 (all out of bounds: the copy fills zeros and still
    // counts its full bytes, so every stage completes on a fixed byte count) past the
    // batch's pages or for a rejected id
    for (int64_t t = cid, i = 0; t < ntiles; t += ncl, ++i) {
      const int r = static_cast<int>(i % kRcRing);
      const bool ok = i < kRcRing ||
                      mbar_wait(&rempty[r], ((i / kRcRing) - 1) & 1, abort_flag, p.dev_err);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (lane < BPC) {
        int32_t y = -kBlockSize;
        const int64_t g = (t / NU) * 2 * BPT + h * BPT + pr * BPC + lane;
        if (g < total) {
          int lo = 0, hi = p.batch;                 // request b with vcum[b] <= g < vcum[b+1]
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.vcum[mid] <= g) lo = mid; else hi = mid;
          }
          const int32_t id = p.block_table[static_cast<int64_t>(lo) * p.bt_stride + (g - p.vcum[lo])];
          if (id >= 0 && id < p.num_blocks) y = id * kBlockSize;
          else if (t % NU == 0) atomicOr(p.dev_err, RCP_DEVERR_BAD_BLOCK);
        }
        rows_s[r * 8 + lane] = y;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rfull[r]);
    }
  } else if (warp == 1 && lane == 0 && h == 0) {
    // ------------------------------------------------------------------- MMAs
    constexpr uint32_t idesc = make_idesc_f16(2 * C::MT, C::NT, false, true);
    int64_t n = 0;
    bool ok = true;
    for (int64_t t = cid, i = 0; ok && t < ntiles; t += ncl, ++i) {
      const int b = static_cast<int>(i & 1);
      // both CTAs' epilogues have read this accumulator's previous tile
      if (i >= 2 && !mbar_wait(&tempty[b], ((i >> 1) - 1) & 1, abort_flag, p.dev_err)) break;
      tc_fence_after();
      const uint32_t dt = tmem + b * C::NT;
      for (int kb = 0; kb < C::KB; ++kb, ++n) {
        const int s = static_cast<int>(n % C::STG);
        if (!mbar_wait(&full[s], (n / C::STG) & 1, abort_flag, p.dev_err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sm + s * L::STAGE);
        const uint32_t b0 = a0 + L::A_BYTES;
#pragma unroll
        for (int k = 0; k < 4; ++k) {   // four K=16 steps per 64-wide k-block
          const uint64_t ad = make_sdesc(a0 + k * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = make_sdesc(b0 + k * 2048, 8192, 1024, kSwizzle128B);
          umma_f16_pair(dt, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit_pair(&empty[s], static_cast<uint16_t>((1u << CL) - 1));   // every CTA
      }
      if (ok) umma_commit_pair(&tfull[b], static_cast<uint16_t>(0x3u << lead));
    }
    // the last commits land before this CTA (and its peer, through the final cluster
    // barrier) goes on
    if (n > 0) mbar_wait_drain(&empty[(n - 1) % C::STG], ((n - 1) / C::STG) & 1);
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------------- epilogue
    // warp w reads TMEM lane quarter w % 4: rows 32 (w % 4) .. of this CTA's 128 keys.  A
    // 64-column chunk goes TMEM -> registers -> the warp's staging buffer (row per lane), then
    // leaves as 8 stores of 4 rows x 128 bytes each.
    const int q = warp & 3, row = q * 32 + lane;
    const uint32_t tarr = map_to_rank(smem_u32(&tempty[0]), lead);
    uint8_t* ebuf = sm + L::EPI_OFF + (warp - 2) * L::EPI_BYTES;
    for (int64_t t = cid, i = 0; t < ntiles; t += ncl, ++i) {
      const int b = static_cast<int>(i & 1);
      // this row's page and whether it holds a token of its sequence in a valid block,
      // resolved before the accumulator is waited for
      const int64_t g = (t / NU) * 2 * BPT + h * BPT + row / kBlockSize;
      const int tok = row % kBlockSize;
      bool keep = false;
      if (g < total) {
        int lo = 0, hi = p.batch;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.vcum[mid] <= g) lo = mid; else hi = mid;
        }
        const int64_t blk = g - p.vcum[lo];
        const int32_t id = p.block_table[static_cast<int64_t>(lo) * p.bt_stride + blk];
        keep = id >= 0 && id < p.num_blocks && blk * kBlockSize + tok < p.seq_lens[lo];
      }
      // the row this lane stores in the copy-out: 4 rows per instruction, 8 lanes per row
      const int orow = lane >> 3, ochunk = lane & 7;
      const int64_t g_first = (t / NU) * 2 * BPT + h * BPT + (q * 32) / kBlockSize;
      if (!__all_sync(0xffffffffu, mbar_wait(&tfull[b], (i >> 1) & 1, abort_flag, p.dev_err)))
        break;
      tc_fence_after();
      const uint32_t trow = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * C::NT;
#pragma unroll 1
      for (int c64 = 0; c64 < C::NT; c64 += 64) {
#pragma unroll
        for (int c16 = 0; c16 < 64; c16 += 16) {
          float v[16];
          tmem_ld16(trow + c64 + c16, v);
          tmem_wait_ld();
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const __half2 hv = keep ? __floats2half2_rn(v[e], v[e + 1]) : __floats2half2_rn(0.f, 0.f);
            w8[e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          const int c0 = c16 / 8;   // first 16-byte chunk of these 16 columns
          *reinterpret_cast<uint4*>(ebuf + lane * 128 + (((c0) ^ (lane & 7)) << 4)) =
              make_uint4(w8[0], w8[1], w8[2], w8[3]);
          *reinterpret_cast<uint4*>(ebuf + lane * 128 + (((c0 + 1) ^ (lane & 7)) << 4)) =
              make_uint4(w8[4], w8[5], w8[6], w8[7]);
        }
        __syncwarp();
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += 4) {
          const int r = r0 + orow;   // row of the warp's 32
          const uint4 val = *reinterpret_cast<const uint4*>(ebuf + r * 128 + ((ochunk ^ (r & 7)) << 4));
          const int64_t gr = g_first + r / kBlockSize;
          if (gr < total)
            *reinterpret_cast<uint4*>(static_cast<__half*>(p.vhat) +
                                      (gr * kBlockSize + r % kBlockSize) * HD +
                                      col_tile(t) * C::NT + c64 + ochunk * 8) = val;
        }
        __syncwarp();   // the buffer is rewritten by the next chunk
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tarr + b * 8);   // this warp is done with buffer b
    }
  }
  tc_fence_before();
  cluster_sync_all();   // no CTA leaves (or frees its columns) while the cluster is busy
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, L::TMEM_COLS);
  }
}

// ------------------------------------------------ quantized pages for prefill
// The prefill kernels read fp16 pages through tensor maps.  For a cache of E4M3 or 4-bit
// pages the reconstructing prefill first widens every page the batch reads (the plan's page
// order, as for V^) into fp16 copies in the workspace and re-addresses the block table to
// them.  E4M3 values are exact in fp16, so the kernels that follow compute the same result
// as on the codes themselves; a 4-bit value becomes fp16(code x scale), one rounding (as in
// the decode's value widening).  A streaming pass: 48 KiB (E4M3) or 25.5 KiB (4-bit) read
// and 96 KiB written per page.
constexpr int kWidenThreads = 256;

__device__ __forceinline__ uint32_t widen_e4m3x2(uint32_t codes) {   // low byte -> low half
  const __half2_raw r =
      __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes & 0xFFFFu), __NV_E4M3);
  return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

template <class S, int FMT>
__global__ void __launch_bounds__(kWidenThreads)
    widen_pages_kernel(const AttnParams p, __half* k16, __half* v16, int32_t* table16) {
  constexpr bool I4 = FMT == RCP_PAGES_INT4;
  constexpr int KN = S::H * kBlockSize * S::RK;    // coefficients of a key page
  constexpr int VN = kBlockSize * S::R;            // coefficients of a value page
  // bytes of a page; E4M3: the codes; 4-bit: codes then fp16 scales
  constexpr int KB8 = I4 ? static_cast<int>(Int4Page<S>::KBYTES) : KN;
  constexpr int VB8 = I4 ? static_cast<int>(Int4Page<S>::VBYTES) : VN;
  // work items: 16 code bytes (E4M3) or 4 code bytes (4-bit), each 8 or 16 B of output
  constexpr int KC = I4 ? KN / 8 : KN / 16, VC = I4 ? VN / 8 : VN / 16;
  static_assert(KN % 16 == 0 && VN % 16 == 0 && S::RK % 8 == 0, "page size");
  __shared__ int64_t s_phys;
  griddep_wait();   // page prefix sums (plan) and the appended chunk are visible
  griddep_launch();
  const int64_t total = p.vcum[p.batch];
  const uint8_t* k8 = static_cast<const uint8_t*>(p.k_pages);
  const uint8_t* v8 = static_cast<const uint8_t*>(p.v_pages);
  for (int64_t g = blockIdx.x; g < total; g += gridDim.x) {   // uniform over the CTA
    if (threadIdx.x == 0) {
      int lo = 0, hi = p.batch;                 // request b with vcum[b] <= g < vcum[b+1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.vcum[mid] <= g) lo = mid; else hi = mid;
      }
      const int64_t j = g - p.vcum[lo];
      const int64_t at = static_cast<int64_t>(lo) * p.bt_stride + j;
      int64_t id = p.block_table[at];
      if (id < 0 || id >= p.num_blocks) {
        atomicOr(p.dev_err, RCP_DEVERR_BAD_BLOCK);
        id = -1;
      }
      table16[at] = id < 0 ? -1 : static_cast<int32_t>(g);
      s_phys = id;
    }
    __syncthreads();
    const int64_t phys = s_phys;
    if (phys >= 0) {
      const uint4* ks = reinterpret_cast<const uint4*>(k8 + phys * KB8);
      const uint4* vs = reinterpret_cast<const uint4*>(v8 + phys * VB8);
      uint4* kd = reinterpret_cast<uint4*>(k16 + g * KN);   // fp16 copies: KN, VN halves
      uint4* vd = reinterpret_cast<uint4*>(v16 + g * VN);
      if constexpr (I4) {
        // 8 coefficients (4 code bytes) of one scale group per item: key groups are the r_k
        // values of a (head, token) row, value groups 64 joint coefficients of a token
        const uint8_t* kb = k8 + phys * KB8;
        const uint8_t* vb = v8 + phys * VB8;
        const __half* ksc = reinterpret_cast<const __half*>(kb + Int4Page<S>::KCODES);
        const __half* vsc = reinterpret_cast<const __half*>(vb + Int4Page<S>::VCODES);
        for (int c = threadIdx.x; c < KC + VC; c += kWidenThreads) {
          const bool key = c < KC;
          const int e0 = (key ? c : c - KC) * 8;           // first coefficient of the item
          const uint32_t raw = *reinterpret_cast<const uint32_t*>((key ? kb : vb) + e0 / 2);
          const __half2 sc = __half2half2(key ? ksc[e0 / S::RK]
                                              : vsc[(e0 / S::R) * (S::R / 64) + (e0 % S::R) / 64]);
          uint4* dst = reinterpret_cast<uint4*>((key ? reinterpret_cast<__half*>(kd)
                                                     : reinterpret_cast<__half*>(vd)) + e0);
          *dst = make_uint4(int4x2_to_half2_bits(raw & 0xFFu, sc),
                            int4x2_to_half2_bits((raw >> 8) & 0xFFu, sc),
                            int4x2_to_half2_bits((raw >> 16) & 0xFFu, sc),
                            int4x2_to_half2_bits(raw >> 24, sc));
        }
      } else {
        for (int c = threadIdx.x; c < KC + VC; c += kWidenThreads) {
          const bool key = c < KC;
          const uint4 raw = key ? ks[c] : vs[c - KC];
          uint4* dst = key ? kd + 2 * c : vd + 2 * (c - KC);
          dst[0] = make_uint4(widen_e4m3x2(raw.x), widen_e4m3x2(raw.x >> 16), widen_e4m3x2(raw.y),
                              widen_e4m3x2(raw.y >> 16));
          dst[1] = make_uint4(widen_e4m3x2(raw.z), widen_e4m3x2(raw.z >> 16), widen_e4m3x2(raw.w),
                              widen_e4m3x2(raw.w >> 16));
        }
      }
    }
    __syncthreads();   // s_phys is rewritten for the next page
  }
}

// --------------------------------------------------------------------------- launches
template <class S>
cudaError_t launch_widen(const AttnParams& p, void* k16, void* v16, int32_t* table16,
                         int64_t max_pages, int num_sms, cudaStream_t stream, bool pdl) {
  if (max_pages <= 0) return cudaSuccess;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;   // grid-stride over the pages
  const unsigned grid = static_cast<unsigned>(max_pages < cap ? max_pages : cap);
  if (p.page_format == RCP_PAGES_INT4)
    return launch_pdl(widen_pages_kernel<S, RCP_PAGES_INT4>, dim3(grid), dim3(kWidenThreads), 0,
                      stream, pdl, p, static_cast<__half*>(k16), static_cast<__half*>(v16),
                      table16);
  return launch_pdl(widen_pages_kernel<S, RCP_PAGES_FP8_E4M3>, dim3(grid), dim3(kWidenThreads), 0,
                    stream, pdl, p, static_cast<__half*>(k16), static_cast<__half*>(v16), table16);
}

template <class S>
cudaError_t prepare_recon() {
  return cudaFuncSetAttribute(recon_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              ReconSmem<S>::ALLOC);
}

// max_pages bounds the pages of the batch (batch x max_blocks_per_seq); CTAs past the
// actual count exit at once.
template <class S>
cudaError_t launch_recon(const CUtensorMap& vp, const CUtensorMap& w_v_mn, const AttnParams& p,
                         int64_t max_pages, int num_sms, cudaStream_t stream, bool pdl) {
  using C = ReconCfg<S>;
  constexpr int CL = 2 * recon_pairs<S>();
  constexpr int64_t PAGES = 2 * C::MT / kBlockSize;   // pages per tile
  const int64_t units = (max_pages + PAGES - 1) / PAGES * (S::H * S::D / C::NT) / (CL / 2);
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kRcThreads);
  cfg.dynamicSmemBytes = ReconSmem<S>::ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // persistent: as many clusters as can be resident at once (the SMs of a GPU partition
  // do not always divide into 4-CTA clusters), queried once
  static int fit = 0;
  if (fit == 0) {
    cfg.gridDim = dim3(static_cast<unsigned>(CL * (num_sms / CL)));
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, recon_kernel<S>, &cfg) != cudaSuccess || n <= 0) {
      (void)cudaGetLastError();   // a failed query leaves no error behind
      n = num_sms / CL;
    }
    fit = n;
  }
  const int64_t clusters = units < fit ? units : fit;
  const int64_t grid = CL * clusters;
  if (grid <= 0) return cudaSuccess;
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, recon_kernel<S>, vp, w_v_mn, p);
}

template cudaError_t prepare_recon<ShapeMain>();
template cudaError_t prepare_recon<ShapeTiny>();
template cudaError_t launch_recon<ShapeMain>(const CUtensorMap&, const CUtensorMap&,
                                             const AttnParams&, int64_t, int, cudaStream_t, bool);
template cudaError_t launch_recon<ShapeTiny>(const CUtensorMap&, const CUtensorMap&,
                                             const AttnParams&, int64_t, int, cudaStream_t, bool);
template cudaError_t launch_widen<ShapeMain>(const AttnParams&, void*, void*, int32_t*, int64_t, int,
                                             cudaStream_t, bool);
template cudaError_t launch_widen<ShapeTiny>(const AttnParams&, void*, void*, int32_t*, int64_t, int,
                                             cudaStream_t, bool);

}  // namespace rcp
