// Split-K combine fused with the W_v up-projection: the decode's third launch, after the
// split-K attention kernel (decode.cu).
//
// The Proxima page ("Kernel profiling breakdown") runs a combine-splits kernel after its
// split-K attention and one matmul per step for the output projection.  Here both are one
// launch.  For a tile of NT requests, a head h and a slice of RANKS value ranks (KSPLIT
// slices cover R), one CTA of 128 threads:
//   1. merges the tile's partial records for head h over its ranks,
//        z_h = sum_i 2^(m_i - M) z_i,h / sum_i 2^(m_i - M) l_i,h,
//      i over the records of the request (one per work partition that touched it), M the
//      largest m_i.  The records' (m, l) groups arrive by one pair of tensor copies and
//      their rank slices stream through a ring of CHUNK-record tensor copies; z lands in
//      shared memory as an fp16 (hi, lo) pair, the B operand of
//   2. D[j][q] = sum_r W_v[r][h*d + j] z_h[q][r] over the CTA's ranks on tcgen05
//      (A = the W_v slice MN-major, fetched before waiting on the split-K kernel, which
//      never writes it), fp32 accumulator in tensor memory;
//   3. stores its fp32 partial D in the workspace; the CTA that completes its (tile, head)
//      group (an atomic counter) adds the KSPLIT partials in slice order (deterministic)
//      and writes o as fp16.  No CTA waits for another, so the grid needs no co-residency.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "rcp.h"
#include "shape.h"

namespace rcp {

constexpr int kCombThreads = 128;
constexpr int kAKb = 128 * 64 * 2;   // one k-block of A: 64 value ranks x 128 head elements

template <class S>
struct CombineSmem {
  using C = CombineCfg<S>;
  static constexpr int NT = C::NT, KB = C::KB, SB = C::RANKS * 4, NW = C::REC_ROWS;
  static constexpr int B_BYTES = NT * 128;                    // one of z_hi / z_lo per k-block
  static constexpr int A_OFF = 0;                             // KB x kAKb, 1024-aligned
  static constexpr int B_OFF = A_OFF + KB * kAKb;             // KB x (hi, lo)
  static constexpr int RING_OFF = B_OFF + KB * 2 * B_BYTES;   // NBUF x CHUNK records x SB
  static constexpr int M_OFF = RING_OFF + C::NBUF * C::CHUNK * SB;   // NW x 4-float m groups
  static constexpr int L_OFF = M_OFF + NW * 16;               // NW x 4-float l groups
  static constexpr int W_OFF = L_OFF + NW * 16;               // NW merge weights
  static constexpr int QI_OFF = (W_OFF + NW * 4 + 15) / 16 * 16;   // NT x int2
  static constexpr int SCR_OFF = QI_OFF + NT * 8;             // kCombThreads x float4
  static constexpr int BAR_OFF = SCR_OFF + kCombThreads * 16;
  static constexpr int NBAR = KB + 2 + C::NBUF;               // A[KB], (m, l), ring[NBUF], acc
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;         // tmem slot, abort, base, last
  static constexpr int TOTAL = MISC_OFF + 32;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr int TMEM_COLS = NT < 32 ? 32 : NT;
  static_assert(B_OFF % 1024 == 0 && B_BYTES % 1024 == 0 && RING_OFF % 128 == 0 &&
                    (C::CHUNK * SB) % 128 == 0 && M_OFF % 128 == 0 && L_OFF % 128 == 0 &&
                    SCR_OFF % 16 == 0 && BAR_OFF % 8 == 0,
                "operand / tensor-copy / float4 / mbarrier alignment");
  static_assert(ALLOC <= 113 * 1024, "two CTAs per SM");
};

template <class S>
__global__ void __launch_bounds__(kCombThreads)
    combine_upproj_kernel(const __grid_constant__ CUtensorMap map_wv,
                          const __grid_constant__ CUtensorMap map_rec,
                          const __grid_constant__ CUtensorMap map_ml, const CombineParams p) {
  using C = CombineCfg<S>;
  using L = CombineSmem<S>;
  constexpr int R = S::R, HP = S::HP, NT = C::NT, KB = C::KB, CH = C::CHUNK, SB = L::SB;
  constexpr int NG = C::RANKS / 4;                  // float4 rank groups
  constexpr int NSET = kCombThreads / NG;           // thread sets
  constexpr int QMAX = NT / NSET;                   // queries per thread
  static_assert(kCombThreads % NG == 0 && NT % NSET == 0, "merge tiling");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* afull = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
  uint64_t* mlbar = afull + KB;
  uint64_t* cbar = mlbar + 1;
  uint64_t* accb = cbar + C::NBUF;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);
  int64_t* base_s = reinterpret_cast<int64_t*>(sm + L::MISC_OFF + 8);
  int* last_s = reinterpret_cast<int*>(sm + L::MISC_OFF + 16);
  const float* m4 = reinterpret_cast<const float*>(sm + L::M_OFF);
  const float* l4 = reinterpret_cast<const float*>(sm + L::L_OFF);
  float* w_s = reinterpret_cast<float*>(sm + L::W_OFF);
  int2* qinfo = reinterpret_cast<int2*>(sm + L::QI_OFF);   // first record id, record count
  float4* scr = reinterpret_cast<float4*>(sm + L::SCR_OFF);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ks = blockIdx.x % C::KSPLIT;              // value-rank slice
  const int h = (blockIdx.x / C::KSPLIT) % S::H;
  const int tile = blockIdx.x / (C::KSPLIT * S::H);
  const int grp = tile * S::H + h;                    // (tile, head) group of KSPLIT CTAs
  const int n0 = tile * NT;
  const int r0 = ks * C::RANKS;
  const int nqt = min(NT, p.nq - n0);                 // real queries of the tile

  if (tid == 0) {
    for (int k = 0; k < KB; ++k) mbar_init(&afull[k], 1);
    mbar_init(mlbar, 1);
    for (int b = 0; b < C::NBUF; ++b) mbar_init(&cbar[b], 1);
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
  // A: the W_v slice, MN-major, two 64 (j) x 64 (r) boxes per k-block; no kernel writes it
  if (tid == 0) {
    prefetch_tmap(&map_wv);
    prefetch_tmap(&map_rec);
    prefetch_tmap(&map_ml);
    for (int k = 0; k < KB; ++k) {
      mbar_arrive_expect_tx(&afull[k], kAKb);
      tma_load_2d(sm + L::A_OFF + k * kAKb, &map_wv, h * S::D, r0 + k * 64, &afull[k]);
      tma_load_2d(sm + L::A_OFF + k * kAKb + kAKb / 2, &map_wv, h * S::D + 64, r0 + k * 64,
                  &afull[k]);
    }
  }
  griddep_wait();   // the records and block prefix sums of the split-K kernel are written
  griddep_launch();

  // ---- (1) record range of every query: one round of loads
  {
    const int64_t T = p.cum[p.nq];
    const int64_t cn0 = p.cum[n0];
    // partitions with blocks (the split-K kernel's rule)
    const int64_t Gm = (T + decode_min_pages<S>(p.nq) - 1) / decode_min_pages<S>(p.nq);
    const int G = static_cast<int>(Gm < p.parts ? Gm : p.parts);
    // the partition whose range [c*T/G, (c+1)*T/G) holds block g
    auto part_of = [&](int64_t g) { return static_cast<int>(((g + 1) * G + T - 1) / T - 1); };
    // record ids of request n are n + first .. n + last partition it touched; over the
    // tile they grow with n, so id - base (base: the tile's first id) indexes the records
    const int64_t base = T > 0 ? n0 + part_of(cn0 < T ? cn0 : T - 1) : 0;
    for (int q = tid; q < NT; q += kCombThreads) {
      int2 qi = make_int2(0, 0);
      if (q < nqt) {
        const int64_t c0 = p.cum[n0 + q], c1 = p.cum[n0 + q + 1];
        if (c1 > c0) {
          const int pf = part_of(c0), pl = part_of(c1 - 1);
          qi = make_int2(static_cast<int>(n0 + q + pf - base), pl - pf + 1);
        }
      }
      qinfo[q] = qi;
    }
    if (tid == 0) *base_s = T > 0 ? base : -1;
  }
  __syncthreads();
  const int64_t base = *base_s;
  int span = 0;   // record ids in use: [0, span); the last query with records ends it
  if (base >= 0)
    for (int q = nqt - 1; q >= 0 && span == 0; --q) span = qinfo[q].x + qinfo[q].y;
  const int nch = (span + CH - 1) / CH;
  // ---- (2) tensor copies: the (m, l) groups of every record, and the first ring chunks
  int issued = 0;   // thread 0: ring chunks requested
  if (tid == 0 && span > 0) {
    const int y = static_cast<int>(base);
    mbar_arrive_expect_tx(mlbar, L::NW * 32);
    tma_load_2d(sm + L::M_OFF, &map_ml, R * HP + (h & ~3), y, mlbar);
    tma_load_2d(sm + L::L_OFF, &map_ml, R * HP + HP + (h & ~3), y, mlbar);
    for (int c = 0; c < C::NBUF && c < nch; ++c, ++issued) {
      mbar_arrive_expect_tx(&cbar[c], CH * SB);
      tma_load_2d(sm + L::RING_OFF + c * CH * SB, &map_rec, h * R + r0, y + c * CH, &cbar[c]);
    }
  }
  // meanwhile: zero B rows past the tile's last query
  for (int i = tid; i < (NT - nqt) * 8 * KB; i += kCombThreads) {
    const int q = nqt + i / (8 * KB), rem = i % (8 * KB);
    uint8_t* st = sm + L::B_OFF + (rem >> 3) * 2 * L::B_BYTES + q * 128 + (rem & 7) * 16;
    *reinterpret_cast<uint4*>(st) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(st + L::B_BYTES) = make_uint4(0, 0, 0, 0);
  }
  bool ok = span == 0 || __syncthreads_and(mbar_wait(mlbar, 0, abort_flag, p.dev_err));
  // ---- (3) merge weights w = 2^(m - M) / sum 2^(m - M) l per query (M its largest m):
  // a warp per query over its records when the tile has few queries (many records each),
  // else a thread per query
  const int hq = h & 3;
  auto weigh = [&](int2 qi, int i0, int step, bool warp_wide) {
    float mx = -INFINITY;
    for (int i = i0; i < qi.y; i += step) mx = fmaxf(mx, m4[(qi.x + i) * 4 + hq]);
    if (warp_wide)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float sum = 0.f;
    for (int i = i0; i < qi.y; i += step) {
      const float m = m4[(qi.x + i) * 4 + hq];
      const float e = m == -INFINITY ? 0.f : exp2f(m - mx);
      w_s[qi.x + i] = e;
      sum = fmaf(e, l4[(qi.x + i) * 4 + hq], sum);
    }
    if (warp_wide)
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    for (int i = i0; i < qi.y; i += step) w_s[qi.x + i] *= inv;
  };
  if (ok) {
    if (nqt <= kCombThreads / 32) {
      if (warp < nqt) weigh(qinfo[warp], lane, 32, true);
    } else {
      for (int q = tid; q < nqt; q += kCombThreads) weigh(qinfo[q], 0, 1, false);
    }
  }
  __syncthreads();
  // ---- (4) z of (query, 4 consecutive ranks g), accumulated chunk by chunk; with fewer
  // queries than thread sets, nsplit sets (a power of two) share each query's records
  const int g = tid % NG, set = tid / NG;
  const int nsplit = nqt >= NSET ? 1 : 1 << (31 - __clz(NSET / nqt));
  const int part = set & (nsplit - 1), qstep = NSET / nsplit, q0 = set / nsplit;
  float4 acc[QMAX];
#pragma unroll
  for (int k = 0; k < QMAX; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c = 0; c < nch; ++c) {
    const int buf = c % C::NBUF;
    ok = __syncthreads_and(ok && mbar_wait(&cbar[buf], (c / C::NBUF) & 1, abort_flag, p.dev_err));
    const uint8_t* chunk = sm + L::RING_OFF + buf * CH * SB + g * 16;
    const int c0 = c * CH, c1 = c0 + CH;
#pragma unroll
    for (int k = 0; k < QMAX; ++k) {
      const int q = q0 + k * qstep;
      if (q >= nqt || !ok) continue;
      const int2 qi = qinfo[q];
      if (qi.x >= c1 || qi.x + qi.y <= c0) continue;   // no record of q in this chunk
      const int hi = min(qi.x + qi.y, c1);
      // this set's records of the query: qi.x + part, then every nsplit-th
      int i = qi.x + part;
      if (i < c0) i += (c0 - i + nsplit - 1) & ~(nsplit - 1);
      for (; i < hi; i += nsplit) {
        const float w = w_s[i];
        const float4 v = *reinterpret_cast<const float4*>(chunk + (i - c0) * SB);
        acc[k].x = fmaf(w, v.x, acc[k].x);
        acc[k].y = fmaf(w, v.y, acc[k].y);
        acc[k].z = fmaf(w, v.z, acc[k].z);
        acc[k].w = fmaf(w, v.w, acc[k].w);
      }
    }
    __syncthreads();   // every thread is done with this chunk's buffer
    if (tid == 0 && ok && c + C::NBUF < nch) {
      mbar_arrive_expect_tx(&cbar[buf], CH * SB);
      tma_load_2d(sm + L::RING_OFF + buf * CH * SB, &map_rec, h * R + r0,
                  static_cast<int>(base) + (c + C::NBUF) * CH, &cbar[buf]);
      ++issued;
    }
  }
  if (!ok && tid == 0 && span > 0) {   // a wait gave up: let the copies in flight land
    mbar_wait_drain(mlbar, 0);
    for (int i = 0; i < issued; ++i) mbar_wait_drain(&cbar[i % C::NBUF], (i / C::NBUF) & 1);
  }
  // z as an fp16 (hi, lo) pair into the B operand: query n, rank c of a k-block at byte
  // n * 128 + ((c / 8) ^ (n % 8)) * 16 + (c % 8) * 2 (K-major, 128-byte swizzle)
  auto store = [&](int q, float4 z) {
    const float zz[4] = {z.x, z.y, z.z, z.w};
    __half hv[4], lv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      hv[e] = __float2half_rn(zz[e]);
      lv[e] = __float2half_rn(zz[e] - __half2float(hv[e]));
    }
    const int rr = g * 4, kb = rr >> 6, cc = rr & 63;
    uint8_t* st = sm + L::B_OFF + kb * 2 * L::B_BYTES;
    const int off = q * 128 + (((cc >> 3) ^ (q & 7)) << 4) + (cc & 7) * 2;
    *reinterpret_cast<uint2*>(st + off) = *reinterpret_cast<const uint2*>(hv);
    *reinterpret_cast<uint2*>(st + L::B_BYTES + off) = *reinterpret_cast<const uint2*>(lv);
  };
  if (nsplit == 1) {
#pragma unroll
    for (int k = 0; k < QMAX; ++k) {
      const int q = set + k * NSET;
      if (q < nqt) store(q, acc[k]);
    }
  } else {
    scr[set * NG + g] = acc[0];
    __syncthreads();
    const int q = q0;
    if (part == 0 && q < nqt) {
      float4 z = acc[0];
      for (int k = 1; k < nsplit; ++k) {   // fixed order: the result does not depend on timing
        const float4 v = scr[(set + k) * NG + g];
        z.x += v.x; z.y += v.y; z.z += v.z; z.w += v.w;
      }
      store(q, z);
    }
  }
  fence_proxy_async_smem();   // generic stores -> the MMA's async-proxy reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---- (5) D = W_v slice^T z over this CTA's ranks (hi and lo parts)
  if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = make_idesc_f16(128, NT, /*a_mn_major=*/true, /*b_mn_major=*/false);
    int kb = 0;
    for (; kb < KB; ++kb) {
      if (!mbar_wait(&afull[kb], 0, abort_flag, p.dev_err)) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(sm + L::A_OFF + kb * kAKb);
      const uint32_t b0 = smem_u32(sm + L::B_OFF + kb * 2 * L::B_BYTES);
#pragma unroll
      for (int k = 0; k < 4; ++k) {   // four K=16 steps per 64-wide k-block
        const uint64_t ad = make_sdesc(a0 + k * 2048, kAKb / 2, 1024, kSwizzle128B);
        umma_f16(tmem, ad, make_sdesc(b0 + k * 32, 16, 1024, kSwizzle128B), idesc,
                 (kb > 0 || k > 0) ? 1u : 0u);
        umma_f16(tmem, ad, make_sdesc(b0 + L::B_BYTES + k * 32, 16, 1024, kSwizzle128B), idesc,
                 1u);
      }
    }
    umma_commit(accb);
    if (kb < KB) {   // an A copy timed out: let the rest land
      mbar_wait_drain(accb, 0);
      for (int k = kb; k < KB; ++k) mbar_wait_drain(&afull[k], 0);
    }
  }
  __syncwarp();
  // ---- (6) the fp32 partial D [col][row] into the workspace (TMEM lane = row = j)
  const bool have_acc = __all_sync(0xffffffffu, mbar_wait(accb, 0, abort_flag, p.dev_err)) && ok;
  tc_fence_after();
  const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int row = warp * 32 + lane;
  float* part_out = p.upart + (static_cast<size_t>(grp) * C::KSPLIT + ks) * NT * 128;
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
    for (int e = 0; e < 16; ++e) part_out[(c0 + e) * 128 + row] = v[e];
  }
  // ---- (7) the last CTA of the (tile, head) group adds the partials in slice order
  __threadfence();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) *last_s = atomicAdd(&p.ucnt[grp], 1) == C::KSPLIT - 1;
  __syncthreads();
  if (*last_s) {
    __threadfence();
    // the tile's real columns only, four rows per float4; UNR positions' loads of every
    // slice are issued before any is added, so the reads overlap
    const float4* parts =
        reinterpret_cast<const float4*>(p.upart + static_cast<size_t>(grp) * C::KSPLIT * NT * 128);
    constexpr int UNR = 4, QUADS = S::D / 4;            // float4 per column
    const int npos = nqt * QUADS;
    for (int i0 = tid; i0 < npos; i0 += kCombThreads * UNR) {
      float4 v[UNR][C::KSPLIT];
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int i = i0 + u * kCombThreads;
        if (i < npos) {
          const int col = i / QUADS, j4 = i % QUADS;
#pragma unroll
          for (int s2 = 0; s2 < C::KSPLIT; ++s2) v[u][s2] = __ldcg(parts + (s2 * NT + col) * 32 + j4);
        }
      }
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        const int i = i0 + u * kCombThreads;
        if (i >= npos) continue;
        float4 o = v[u][0];
#pragma unroll
        for (int s2 = 1; s2 < C::KSPLIT; ++s2) {   // slice order: deterministic
          o.x += v[u][s2].x; o.y += v[u][s2].y; o.z += v[u][s2].z; o.w += v[u][s2].w;
        }
        const int col = i / QUADS, j4 = i % QUADS;
        const __half2 a = __floats2half2_rn(o.x, o.y), b = __floats2half2_rn(o.z, o.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&a);
        w.y = *reinterpret_cast<const uint32_t*>(&b);
        *reinterpret_cast<uint2*>(static_cast<__half*>(p.out) +
                                  (static_cast<size_t>(n0 + col) * S::H + h) * S::D + j4 * 4) = w;
      }
    }
    if (tid == 0) p.ucnt[grp] = 0;   // ready for the next call (also cleared per call)
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <class S>
cudaError_t prepare_combine() {
  return cudaFuncSetAttribute(combine_upproj_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              CombineSmem<S>::ALLOC);
}

template <class S>
cudaError_t launch_combine_upproj(const CUtensorMap& w_v_mn, const CUtensorMap& rec_slices,
                                  const CUtensorMap& rec_ml, const CombineParams& p,
                                  cudaStream_t stream, bool pdl) {
  using C = CombineCfg<S>;
  const int tiles = (p.nq + C::NT - 1) / C::NT;
  return launch_pdl(combine_upproj_kernel<S>, dim3(tiles * S::H * C::KSPLIT), dim3(kCombThreads),
                    CombineSmem<S>::ALLOC, stream, pdl, w_v_mn, rec_slices, rec_ml, p);
}

template cudaError_t prepare_combine<ShapeMain>();
template cudaError_t prepare_combine<ShapeTiny>();
template cudaError_t launch_combine_upproj<ShapeMain>(const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, const CombineParams&,
                                                      cudaStream_t, bool);
template cudaError_t launch_combine_upproj<ShapeTiny>(const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, const CombineParams&,
                                                      cudaStream_t, bool);

}  // namespace rcp
