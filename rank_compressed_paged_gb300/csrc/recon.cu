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
// vcum), are the rows of one GEMM D[keys x H*d] = C_v[keys x R] * W_v[R x H*d]:
//   * one CTA per (128 keys = 8 pages, 256 columns): A = the 8 pages' C_v rows, one
//     16 x 64 tensor-map box per page per 64-wide k-block (K-major, 128-byte swizzle);
//     B = W_v[k-block rows, 256 columns], four 64 x 64 boxes (MN-major);
//   * tcgen05.mma M=128, N=256, K=16 steps into a 256-column TMEM accumulator, two
//     pipeline stages; two CTAs share an SM so one's epilogue overlaps the other's loop;
//   * the epilogue writes V^ rows as fp16, zero for the slots of a page past the end of
//     its sequence (so that the attention can never meet 0 * NaN there).
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

constexpr int kRcThreads = 128;   // warp 0 copies, warp 1 MMAs, all four the epilogue

template <class S>
struct ReconSmem {
  using C = ReconCfg<S>;
  static constexpr int A_BYTES = C::MT * 128;          // 128 keys x 64 ranks
  static constexpr int B_BYTES = C::NT * 128;          // 64 ranks x 256 columns
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = C::STG * STAGE;       // full[STG], empty[STG], acc
  static constexpr int INFO_OFF = BAR_OFF + (2 * C::STG + 1) * 8;   // [8] valid tokens / page
  static constexpr int MISC_OFF = INFO_OFF + 8 * 4;    // tmem slot, abort flag
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr int TMEM_COLS = C::NT;
  static_assert(STAGE % 1024 == 0, "stages keep 1024-byte alignment");
  static_assert(2 * ALLOC <= 228 * 1024, "two CTAs per SM");
};

template <class S>
__global__ void __launch_bounds__(kRcThreads, 2)
    recon_kernel(const __grid_constant__ CUtensorMap vp_map, const __grid_constant__ CUtensorMap w_map,
                 const AttnParams p) {
  using C = ReconCfg<S>;
  using L = ReconSmem<S>;
  constexpr int HD = S::H * S::D, NTN = HD / C::NT, BPT = C::MT / kBlockSize;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
  uint64_t* empty = full + C::STG;
  uint64_t* accb = empty + C::STG;
  int* valid_s = reinterpret_cast<int*>(sm + L::INFO_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x / NTN, nt = blockIdx.x % NTN;   // CTAs of one key tile adjacent

  griddep_wait();   // page prefix sums (plan) and the appended chunk are visible
  griddep_launch();
  const int64_t total = p.vcum[p.batch];
  const int64_t g0 = static_cast<int64_t>(tile) * BPT;       // first page of the tile
  if (g0 >= total) return;                                   // uniform over the CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STG; ++s) {
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

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ copies
    prefetch_tmap(&vp_map);
    prefetch_tmap(&w_map);
    int32_t phys[BPT];
    int nload = 0;
#pragma unroll
    for (int jb = 0; jb < BPT; ++jb) {
      const int64_t g = g0 + jb;
      int32_t id = -1, nvalid = 0;
      if (g < total) {
        int lo = 0, hi = p.batch;                 // request b with vcum[b] <= g < vcum[b+1]
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (p.vcum[mid] <= g) lo = mid; else hi = mid;
        }
        const int64_t blk = g - p.vcum[lo];
        id = p.block_table[static_cast<int64_t>(lo) * p.bt_stride + blk];
        if (id < 0 || id >= p.num_blocks) {
          atomicOr(p.dev_err, RCP_DEVERR_BAD_BLOCK);
          id = -1;
        } else {
          const int64_t left = p.seq_lens[lo] - blk * kBlockSize;
          nvalid = static_cast<int32_t>(left < kBlockSize ? left : kBlockSize);
        }
      }
      phys[jb] = id;
      valid_s[jb] = nvalid;
      nload += id >= 0;
    }
    int issued = 0;
    for (int kb = 0; kb < C::KB; ++kb) {
      const int s = kb % C::STG;
      if (kb >= C::STG &&
          !mbar_wait(&empty[s], ((kb / C::STG) - 1) & 1, abort_flag, p.dev_err))
        break;
      uint8_t* st = sm + s * L::STAGE;
      mbar_arrive_expect_tx(&full[s], nload * 2048 + L::B_BYTES);
#pragma unroll
      for (int jb = 0; jb < BPT; ++jb)
        if (phys[jb] >= 0)
          tma_load_2d(st + jb * 2048, &vp_map, kb * 64, phys[jb] * kBlockSize, &full[s]);
#pragma unroll
      for (int q = 0; q < C::NT / 64; ++q)
        tma_load_2d(st + L::A_BYTES + q * 8192, &w_map, nt * C::NT + q * 64, kb * 64, &full[s]);
      ++issued;
    }
    if (*abort_flag)
      for (int i = (issued > C::STG ? issued - C::STG : 0); i < issued; ++i)
        mbar_wait_drain(&full[i % C::STG], (i / C::STG) & 1);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------- MMAs
    constexpr uint32_t idesc = make_idesc_f16(128, C::NT, false, true);
    int kb = 0;
    for (; kb < C::KB; ++kb) {
      const int s = kb % C::STG;
      if (!mbar_wait(&full[s], (kb / C::STG) & 1, abort_flag, p.dev_err)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sm + s * L::STAGE);
      const uint32_t b0 = a0 + L::A_BYTES;
#pragma unroll
      for (int k = 0; k < 4; ++k) {   // four K=16 steps per 64-wide k-block
        const uint64_t ad = make_sdesc(a0 + k * 32, 16, 1024, kSwizzle128B);
        const uint64_t bd = make_sdesc(b0 + k * 2048, 8192, 1024, kSwizzle128B);
        umma_f16(tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(accb);
    if (kb < C::KB) mbar_wait_drain(accb, 0);
  }
  __syncwarp();
  __syncthreads();   // valid_s is written

  // ------------------------------------------------------------------- epilogue
  // TMEM lane = key row of the tile; warp-uniform guards around the collective loads
  const bool have = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, p.dev_err));
  tc_fence_after();
  const int row = warp * 32 + lane;
  const int64_t g = g0 + row / kBlockSize;
  const bool in_range = g < total;
  const bool keep = row % kBlockSize < valid_s[row / kBlockSize];
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  __half* dst = static_cast<__half*>(p.vhat) + (g * kBlockSize + row % kBlockSize) * HD + nt * C::NT;
#pragma unroll 1
  for (int c0 = 0; c0 < C::NT; c0 += 16) {
    float v[16];
    if (have) {
      tmem_ld16(trow + c0, v);
      tmem_wait_ld();
    }
    uint32_t w8[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const __half2 hv = (have && keep) ? __floats2half2_rn(v[e], v[e + 1])
                                        : __floats2half2_rn(0.f, 0.f);
      w8[e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    if (in_range) {
      *reinterpret_cast<uint4*>(dst + c0) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
      *reinterpret_cast<uint4*>(dst + c0 + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
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
                         int64_t max_pages, cudaStream_t stream, bool pdl) {
  using C = ReconCfg<S>;
  const int64_t tiles = (max_pages + C::MT / kBlockSize - 1) / (C::MT / kBlockSize);
  const int64_t grid = tiles * (S::H * S::D / C::NT);
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  return launch_pdl(recon_kernel<S>, dim3(static_cast<unsigned>(grid)), dim3(kRcThreads),
                    ReconSmem<S>::ALLOC, stream, pdl, vp, w_v_mn, p);
}

template cudaError_t prepare_recon<ShapeMain>();
template cudaError_t prepare_recon<ShapeTiny>();
template cudaError_t launch_recon<ShapeMain>(const CUtensorMap&, const CUtensorMap&,
                                             const AttnParams&, int64_t, cudaStream_t, bool);
template cudaError_t launch_recon<ShapeTiny>(const CUtensorMap&, const CUtensorMap&,
                                             const AttnParams&, int64_t, cudaStream_t, bool);
template cudaError_t launch_widen<ShapeMain>(const AttnParams&, void*, void*, int32_t*, int64_t, int,
                                             cudaStream_t, bool);
template cudaError_t launch_widen<ShapeTiny>(const AttnParams&, void*, void*, int32_t*, int64_t, int,
                                             cudaStream_t, bool);

}  // namespace rcp
