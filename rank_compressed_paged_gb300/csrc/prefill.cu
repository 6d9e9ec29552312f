// Chunked-prefill attention over low-rank paged coefficients on tensor cores.
//
// The "Per-prefill-chunk attention" step of the Proxima page: every row i of a request's
// chunk (absolute position P + i) attends keys 0 .. P + i of the paged cache, after the
// chunk itself has been appended.  The scores are rank-space products and the values a
// joint coefficient contraction, so one CTA owns (request, head h, 128 query rows, one
// slice of up to 256 of the R joint ranks) and walks the causal key range in tiles of
// 128 tokens (8 pages):
//
//   S   = Q~_h C_k,h^T          tcgen05, M=128 rows x N=128 keys x K=64 (q~ as fp16 hi+lo)
//   P   = exp2(S - m)           one thread per query row (TMEM lane), lazy rescaling
//   Z  += P C_v[:, slice]       tcgen05, M=128 x N=256 x K=128, accumulator in TMEM
//
// S is double-buffered in TMEM so the score MMA of tile j+1 overlaps the softmax of tile
// j, and the softmax of tile j overlaps the value MMA of tile j-1.  At the end each row
// is normalised, split into an fp16 (hi, lo) pair and multiplied by the slice's rows of
// W_v[:, h*d:(h+1)*d] (tcgen05 again); the slices of one (request, head, tile) form a
// thread-block cluster and sum their partial outputs through distributed shared memory.
//
// The reconstructing variant (RECON) attends V^ = C_v W_v rows of head h, rebuilt once per
// key by the reconstruction GEMM: O += P V^_h (M=128 x N=d x K=128) in TMEM, no rank slices,
// and the softmax warps write O / l straight to the output; its key/value ring has three
// stages, and P stays in tensor memory (two buffers, stored by the softmax threads with
// tcgen05.st and read as the value MMA's A operand).
//
// Warps: 0 copies queries and key tiles, 6 copies value tiles and the W_v slice (two
// independent streams: a key stage is freed by its score MMA, a value stage by its value
// MMA), 1 issues the MMAs (and owns TMEM), 2-5 run the softmax and the epilogue (warp w
// serves TMEM lanes 32*(w%4) .. +31).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "rcp.h"
#include "shape.h"

namespace rcp {

constexpr int kPfThreads = 224;   // 0 key copies, 1 MMAs, 2-5 softmax, 6 value copies
constexpr float kPfRescale = 8.f;   // log2 units: weights stay below 2^8 between rescales

// RECON: the values are the reconstructed V^ rows of head h (N = d) instead of a slice
// of the joint coefficients (N = RQ), and the epilogue writes O directly.
template <class S, bool RECON>
struct PfSmem {
  using C = PrefillCfg<S>;
  static constexpr int VN = RECON ? S::D : C::RQ;       // value MMA N
  static constexpr int NQ = RECON ? 1 : C::NQ;          // CTAs per (tile, head)
  static constexpr int NG = VN / 64;                    // 64-wide groups of the value tile
  static constexpr int Q_BYTES = 128 * 128;             // one [128][64] fp16 operand
  static constexpr int K_BYTES = C::KT * 128;           // key coefficients of one tile
  static constexpr int V_BYTES = C::KT * VN * 2;        // value tile
  static constexpr int STAGE = K_BYTES + V_BYTES;
  static constexpr int NS = RECON ? 3 : 2;              // key/value pipeline stages
  // RECON keeps P in tensor memory (two buffers at columns P_TM and P_TM + KT/2, the A
  // operand of the value MMA); the rank-space variant stages it in shared memory
  static constexpr int P_BYTES = RECON ? 0 : 128 * C::KT * 2;
  static constexpr int P_TM = 256 + VN;
  static constexpr int ST_OFF = 2 * Q_BYTES;            // q~ hi at 0, q~ lo at Q_BYTES
  static constexpr int P_OFF = ST_OFF + NS * STAGE;
  static constexpr int ZH_OFF = ST_OFF;                 // epilogue reuses the stage memory
  static constexpr int ZL_OFF = ZH_OFF + 128 * C::RQ * 2;
  static constexpr int W_OFF = ZL_OFF + 128 * C::RQ * 2;
  static constexpr int W_BYTES = C::RQ * S::D * 2;
  static constexpr int END = (RECON || P_OFF + P_BYTES > W_OFF + W_BYTES) ? P_OFF + P_BYTES
                                                                             : W_OFF + W_BYTES;
  static constexpr int NBAR = 11 + 4 * NS;
  static constexpr int BAR_OFF = END;                   // NBAR mbarriers
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;   // tmem slot, abort flag
  static constexpr int TOTAL = MISC_OFF + 16;
  static constexpr int ALLOC = TOTAL + 1024;
  static constexpr int RPC = 128 / NQ;                  // output rows each slice CTA sums
  static constexpr int TMEM_COLS = pow2_at_least(256 + VN, 32);
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(NQ == 1 || NQ * RPC * S::D * 4 <= 2 * 128 * C::RQ * 2, "receive buffer");
  static_assert(256 + VN <= 512 && S::D <= 128, "tensor memory budget");
  static_assert(!RECON || P_TM + C::KT <= TMEM_COLS, "P buffers in tensor memory");
};

template <class S, bool RECON>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qhi_map,
                   const __grid_constant__ CUtensorMap qlo_map,
                   const __grid_constant__ CUtensorMap kp_map,
                   const __grid_constant__ CUtensorMap vp_map,
                   const __grid_constant__ CUtensorMap w_map, const AttnParams p) {
  using C = PrefillCfg<S>;
  using L = PfSmem<S, RECON>;
  constexpr int KT = C::KT, RQ = C::RQ, NQ = L::NQ, NG = L::NG, VN = L::VN, D = S::D, H = S::H;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
  constexpr int NS = L::NS;
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;              // [NS] key half of a stage landed
  uint64_t* v_full = k_full + NS;           // [NS] value half of a stage landed
  uint64_t* k_empty = v_full + NS;          // [NS] score MMA of the stage's tile done
  uint64_t* v_empty = k_empty + NS;         // [NS] value MMA of the stage's tile done
  uint64_t* s_full = v_empty + NS;          // [2] scores of a tile in TMEM
  uint64_t* p_full = s_full + 2;            // [2] softmax weights written (4 warps)
  uint64_t* pv_done = p_full + 2;           // [2] value MMA of a P buffer done
  uint64_t* acc_done = pv_done + 2;
  uint64_t* zq_full = acc_done + 1;
  uint64_t* w_full = zq_full + 1;
  uint64_t* o_done = w_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  griddep_wait();            // plan and rank-space queries are ready
  griddep_launch();
  const int slot = blockIdx.x / (H * NQ);
  const int h = (blockIdx.x / NQ) % H;
  const int slice = blockIdx.x % NQ;                    // cluster rank when NQ > 1
  if (slot >= *p.tcount) return;                        // uniform over the cluster
  const int b = p.tile_b[slot], qt = p.tile_qt[slot];
  const int c0 = p.cu_chunk[b], n = p.cu_chunk[b + 1] - c0;
  const int Lb = p.seq_lens[b], P0 = Lb - n;
  const int i0 = qt * 128;                              // first chunk row of this tile
  const int i_last = min(n, i0 + 128) - 1;
  const int nkt = (P0 + i_last + 1 + KT - 1) / KT;      // key tiles (causal limit)
  const int nblk = (Lb + kBlockSize - 1) / kBlockSize;
  const int row0 = c0 + i0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(acc_done, 1);
    mbar_init(zq_full, 4);
    mbar_init(w_full, 1);
    mbar_init(o_done, 1);
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
  if constexpr (NQ > 1) cluster_sync_all();   // peers are running before any remote store

  if (warp == 0) {
    // ------------------------------------------------------------------ key copies
    // The whole warp: lane jb < 8 resolves page jb of each tile one tile ahead and issues
    // that page's copy (the eight small copies of a tile set the kernel's pace when one
    // thread issues them in turn); lane 0 waits for the stage and arms its byte count.
    constexpr int BPT = KT / kBlockSize;                  // pages per key tile
    if (lane == 0) {
      prefetch_tmap(&kp_map);
      mbar_arrive_expect_tx(q_full, 2 * L::Q_BYTES);
      tma_load_2d(sm, &qhi_map, h * 64, row0, q_full);
      tma_load_2d(sm + L::Q_BYTES, &qlo_map, h * 64, row0, q_full);
    }
    const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
    int32_t nxt = (lane < BPT && lane < nblk) ? table[lane] : -1;
    for (int j = 0; j < nkt; ++j) {
      const int s = j % NS;
      const bool mine = lane < BPT && j * BPT + lane < nblk;
      int32_t phys = mine ? nxt : -1;
      if (mine && (phys < 0 || phys >= p.num_blocks)) {
        atomicOr(p.dev_err, RCP_DEVERR_BAD_BLOCK);
        phys = -1;
      }
      const int nb = (j + 1) * BPT + lane;                 // the next tile's page, in flight
      nxt = (lane < BPT && nb < nblk) ? table[nb] : -1;
      const int nload = __popc(__ballot_sync(0xffffffffu, phys >= 0));
      bool ok = true;
      if (lane == 0) {
        ok = j < NS || mbar_wait(&k_empty[s], ((j / NS) - 1) & 1, abort_flag, p.dev_err);
        if (ok) mbar_arrive_expect_tx(&k_full[s], nload * 2048);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;   // the byte count is armed first
      if (phys >= 0)
        tma_load_2d(sm + L::ST_OFF + s * L::STAGE + lane * 2048, &kp_map, 0,
                    (phys * H + h) * kBlockSize, &k_full[s]);
    }
  } else if (warp == 6) {
    // ---------------------------------------------------------------- value copies
    if constexpr (RECON) {
      // V^ rows of the request are contiguous: one 64-column box of 128 keys per group
      if (lane == 0) {
        prefetch_tmap(&vp_map);
        for (int j = 0; j < nkt; ++j) {
          const int s = j % NS;
          uint8_t* vst = sm + L::ST_OFF + s * L::STAGE + L::K_BYTES;
          if (j >= NS && !mbar_wait(&v_empty[s], ((j / NS) - 1) & 1, abort_flag, p.dev_err)) break;
          mbar_arrive_expect_tx(&v_full[s], NG * KT * 128);
          const int64_t vrow = p.vcum[b] * kBlockSize + static_cast<int64_t>(j) * KT;
#pragma unroll
          for (int g = 0; g < NG; ++g)
            tma_load_2d(vst + g * KT * 128, &vp_map, h * D + g * 64, static_cast<int32_t>(vrow),
                        &v_full[s]);
        }
      }
    } else {
      // the value rank slice of each page: lane jb < 8 resolves page jb of each tile one
      // tile ahead and issues its NG boxes, as the key copies
      constexpr int BPT = KT / kBlockSize;
      if (lane == 0) prefetch_tmap(&vp_map);
      const int32_t* table = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
      int32_t nxt = (lane < BPT && lane < nblk) ? table[lane] : -1;
      for (int j = 0; j < nkt; ++j) {
        const int s = j % NS;
        const bool mine = lane < BPT && j * BPT + lane < nblk;
        const int32_t id = mine ? nxt : -1;
        const int32_t phys = (id >= 0 && id < p.num_blocks) ? id : -1;   // keys report bad ids
        const int nb = (j + 1) * BPT + lane;
        nxt = (lane < BPT && nb < nblk) ? table[nb] : -1;
        const int nload = __popc(__ballot_sync(0xffffffffu, phys >= 0));
        bool go = true;
        if (lane == 0) {
          go = j < NS || mbar_wait(&v_empty[s], ((j / NS) - 1) & 1, abort_flag, p.dev_err);
          if (go) mbar_arrive_expect_tx(&v_full[s], nload * NG * 2048);
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) break;
        uint8_t* vst = sm + L::ST_OFF + s * L::STAGE + L::K_BYTES;
        if (phys >= 0) {
#pragma unroll
          for (int g = 0; g < NG; ++g)
            tma_load_2d(vst + (g * BPT + lane) * 2048, &vp_map, slice * RQ + g * 64,
                        phys * kBlockSize, &v_full[s]);
        }
      }
      // the W_v rows of this slice, into stage memory once every value MMA is done
      if (lane == 0 && mbar_wait(acc_done, 0, abort_flag, p.dev_err)) {
        mbar_arrive_expect_tx(w_full, L::W_BYTES);
        uint8_t* wst = sm + L::W_OFF;
        for (int g = 0; g < D / 64; ++g)
          for (int kb = 0; kb < RQ / 64; ++kb)
            tma_load_2d(wst + (g * (RQ / 64) + kb) * 8192, &w_map, h * D + g * 64,
                        slice * RQ + kb * 64, w_full);
        mbar_wait_drain(w_full, 0);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------------- MMAs
    // Issues whichever MMA is ready (non-blocking probes): the score MMA of tile js once
    // its keys landed and the softmax of tile js-2 released that S buffer, the value MMA
    // of tile jp once its weights are written and its values landed.  The tensor pipe
    // runs them in order, so S(j+1) overlaps the softmax of tile j and PV(j) overlaps
    // the softmax of tile j+1.
    if (lane == 0) {
      constexpr uint32_t id_s = make_idesc_f16(128, KT, false, false);
      constexpr uint32_t id_pv = make_idesc_f16(128, VN, false, true);
      constexpr uint32_t id_o = make_idesc_f16(128, D, false, true);
      const uint32_t qa = smem_u32(sm);
      const uint32_t pa = smem_u32(sm + L::P_OFF);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.dev_err);
      int js = 0, jp = 0;
      uint64_t t_idle = 0;
      while (ok && jp < nkt) {
        bool progress = false;
        if (js < nkt && js <= jp + 1 && mbar_test_wait(&k_full[js % NS], (js / NS) & 1)) {
          tc_fence_after();
          const uint32_t ka = smem_u32(sm + L::ST_OFF + (js % NS) * L::STAGE);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = make_sdesc(ka + kk * 32, 16, 1024, kSwizzle128B);
            umma_f16(tmem + (js & 1) * 128, make_sdesc(qa + kk * 32, 16, 1024, kSwizzle128B), bd,
                     id_s, kk > 0 ? 1u : 0u);
            umma_f16(tmem + (js & 1) * 128,
                     make_sdesc(qa + L::Q_BYTES + kk * 32, 16, 1024, kSwizzle128B), bd, id_s, 1u);
          }
          umma_commit(&s_full[js & 1]);
          umma_commit(&k_empty[js % NS]);
          ++js;
          progress = true;
        }
        // RECON: P buffer jp & 1, each with its own barriers; rank space: one P buffer
        const int pb = RECON ? (jp & 1) : 0;
        const uint32_t pph = RECON ? (jp >> 1) & 1 : jp & 1;
        if (jp < js && mbar_test_wait(&p_full[pb], pph) &&
            mbar_test_wait(&v_full[jp % NS], (jp / NS) & 1)) {
          tc_fence_after();
          const uint32_t va = smem_u32(sm + L::ST_OFF + (jp % NS) * L::STAGE + L::K_BYTES);
#pragma unroll
          for (int ks = 0; ks < KT / 16; ++ks) {
            const uint64_t bd = make_sdesc(va + ks * 2048, (KT / kBlockSize) * 2048, 1024,
                                           kSwizzle128B);
            if constexpr (RECON) {
              umma_f16_ta(tmem + 256, tmem + L::P_TM + pb * (KT / 2) + ks * 8, bd, id_pv,
                          (jp > 0 || ks > 0) ? 1u : 0u);
            } else {
              const uint64_t ad = make_sdesc(pa + (ks >> 2) * 16384 + (ks & 3) * 32, 16, 1024,
                                             kSwizzle128B);
              umma_f16(tmem + 256, ad, bd, id_pv, (jp > 0 || ks > 0) ? 1u : 0u);
            }
          }
          umma_commit(&pv_done[pb]);
          umma_commit(&v_empty[jp % NS]);
          ++jp;
          progress = true;
        }
        if (progress) {
          t_idle = 0;
        } else if (*abort_flag) {
          ok = false;
        } else if (t_idle == 0) {
          t_idle = globaltimer_ns();
        } else if (globaltimer_ns() - t_idle > kWaitLimitNs) {
          *abort_flag = 1;
          atomicOr(p.dev_err, RCP_DEVERR_TIMEOUT);
          ok = false;
        }
      }
      umma_commit(acc_done);
      // up-projection of this slice: O = (z_hi + z_lo) W_v[slice rows, h*d:(h+1)*d]
      if (!RECON && mbar_wait(zq_full, 0, abort_flag, p.dev_err) &&
          mbar_wait(w_full, 0, abort_flag, p.dev_err)) {
        tc_fence_after();
        const uint32_t zh = smem_u32(sm + L::ZH_OFF), zl = smem_u32(sm + L::ZL_OFF);
        const uint32_t wa = smem_u32(sm + L::W_OFF);
#pragma unroll 1
        for (int ks = 0; ks < RQ / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * 16384 + (ks & 3) * 32;
          const uint64_t bd = make_sdesc(wa + ks * 2048, (RQ / 64) * 8192, 1024, kSwizzle128B);
          umma_f16(tmem, make_sdesc(zh + koff, 16, 1024, kSwizzle128B), bd, id_o, ks > 0 ? 1u : 0u);
          umma_f16(tmem, make_sdesc(zl + koff, 16, 1024, kSwizzle128B), bd, id_o, 1u);
        }
      }
      if (!RECON) {
        umma_commit(o_done);
        mbar_wait_drain(o_done, 0);
      }
    }
  } else {
    // ----------------------------------------------- softmax (one thread per query row)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                  // query row within the tile
    const int ci = i0 + r;                              // chunk row
    const bool row_ok = ci < n;
    const int pos = P0 + ci;                            // keys 0 .. pos are attended
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float m_run = -INFINITY, l_run = 0.f;
    uint8_t* pbuf = sm + L::P_OFF;
    for (int j = 0; j < nkt; ++j) {
      const int s = j & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&s_full[s], (j >> 1) & 1, abort_flag, p.dev_err));
      tc_fence_after();
      const int lim = row_ok ? pos - j * KT : -1;       // columns 0 .. lim are valid
      // the whole 128-column score row: eight loads in flight, one wait
      float sv[KT];
      if (ok) {
#pragma unroll
        for (int c = 0; c < KT; c += 16)
          tmem_ld16(tl + s * 128 + c, *reinterpret_cast<float(*)[16]>(&sv[c]));
        tmem_wait_ld();
      }
      const bool full_tile = __all_sync(0xffffffffu, lim >= KT - 1);   // below the diagonal
      // masked columns (diagonal tiles, rows past the chunk, a failed wait) become -inf, so
      // the max and the exponentials below need no per-element test (exp2(-inf) = 0)
      if (!ok || !full_tile) {
#pragma unroll
        for (int c = 0; c < KT; ++c) sv[c] = (ok && c <= lim) ? sv[c] : -INFINITY;
      }
      // row max: four independent chains of three-input maxima
      float mx;
      {
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < KT; c += 8) {
          m4[0] = max3f(m4[0], sv[c], sv[c + 1]);
          m4[1] = max3f(m4[1], sv[c + 2], sv[c + 3]);
          m4[2] = max3f(m4[2], sv[c + 4], sv[c + 5]);
          m4[3] = max3f(m4[3], sv[c + 6], sv[c + 7]);
        }
        mx = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      }
      const float m_new = (mx > m_run + kPfRescale) ? mx : m_run;
      const float alpha = (m_new == m_run) ? 1.f : fast_exp2(m_run - m_new);
      uint32_t packed[KT / 2];
      float rsum;
      {
        const float msub = (m_new == -INFINITY) ? 0.f : m_new;   // rows with no valid key
        const float2 msub2 = make_float2(msub, msub);
        float2 s4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) s4[q] = make_float2(0.f, 0.f);
        // the row sum is taken in fp32 before the weights are rounded to fp16; pairs of
        // columns go through the packed fp32x2 add / subtract
#pragma unroll
        for (int c = 0; c < KT; c += 2) {
          const float2 d = sub_f32x2(make_float2(sv[c], sv[c + 1]), msub2);
          const float2 pp = make_float2(fast_exp2(d.x), fast_exp2(d.y));
          s4[(c >> 1) & 3] = add_f32x2(s4[(c >> 1) & 3], pp);
          const __half2 hp = __floats2half2_rn(pp.x, pp.y);
          packed[c / 2] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        const float2 t2 = add_f32x2(add_f32x2(s4[0], s4[1]), add_f32x2(s4[2], s4[3]));
        rsum = t2.x + t2.y;
      }
      // rank space: the previous tile's value MMA must be done before P is overwritten or
      // Z rescaled.  RECON: P buffer j & 1 must be free (value MMA of tile j-2), and only a
      // rescale needs the previous tile's value MMA
      const bool rescale = __any_sync(0xffffffffu, ok && alpha != 1.f && j > 0);
      if constexpr (RECON) {
        if (j >= 2) ok = mbar_wait(&pv_done[j & 1], ((j - 2) >> 1) & 1, abort_flag, p.dev_err) && ok;
        if (rescale)
          ok = mbar_wait(&pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, p.dev_err) && ok;
      } else {
        if (j > 0) ok = mbar_wait(&pv_done[0], (j - 1) & 1, abort_flag, p.dev_err) && ok;
      }
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      // tcgen05.ld / st are warp-collective: the whole warp rescales when any lane needs it
      // (lanes whose max did not move multiply by 1)
      if (ok && rescale) {
#pragma unroll 1
        for (int c = 0; c < VN; c += 32) {
          float v[16], w[16];
          tmem_ld16(tl + 256 + c, v);
          tmem_ld16(tl + 256 + c + 16, w);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            v[e] *= alpha;
            w[e] *= alpha;
          }
          tmem_st16(tl + 256 + c, v);
          tmem_st16(tl + 256 + c + 16, w);
        }
        tmem_wait_st();
      }
      if constexpr (RECON) {
        // P row r into tensor memory lane r: column c holds keys 2c and 2c+1
        if (ok) {
#pragma unroll
          for (int c = 0; c < KT / 2; c += 16) tmem_st16u(tl + L::P_TM + (j & 1) * (KT / 2) + c, &packed[c]);
          tmem_wait_st();
        }
      } else {
        // P row r, K-major, 128-byte swizzle: 16-byte chunk c of the row sits at c ^ (r % 8)
#pragma unroll
        for (int ch = 0; ch < KT / 8; ++ch) {
          const int kb = ch >> 3, cc = ch & 7;
          *reinterpret_cast<uint4*>(pbuf + kb * 16384 + r * 128 + ((cc ^ (r & 7)) << 4)) =
              make_uint4(packed[ch * 4], packed[ch * 4 + 1], packed[ch * 4 + 2], packed[ch * 4 + 3]);
        }
      }
      l_run = l_run * alpha + rsum;
      m_run = m_new;
      if (j * KT + KT > Lb) {
        // tokens past the end of the request: zero their value rows so that whatever the
        // slots hold (or stale bytes of skipped pages) never meet a zero weight as 0 * NaN
        ok = mbar_wait(&v_full[j % NS], (j / NS) & 1, abort_flag, p.dev_err) && ok;
        uint8_t* vst = sm + L::ST_OFF + (j % NS) * L::STAGE + L::K_BYTES;
        const int first = Lb - j * KT > 0 ? Lb - j * KT : 0;
        const int nrow = KT - first;
        for (int idx = threadIdx.x - 64; idx < nrow * NG * 8; idx += 128) {   // warps 2-5
          const int tok = first + idx / (NG * 8);
          const int rem = idx % (NG * 8);
          const int g = rem >> 3, ch = rem & 7;
          *reinterpret_cast<uint4*>(vst + (g * (KT / kBlockSize) + tok / kBlockSize) * 2048 +
                                    (tok % kBlockSize) * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[RECON ? (j & 1) : 0]);
    }
    const bool ok = __all_sync(0xffffffffu, mbar_wait(acc_done, 0, abort_flag, p.dev_err));
    tc_fence_after();
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    if constexpr (RECON) {
      // ------------------------------------------- O / l straight to the output rows
      if (ok) {   // warp-uniform: every lane loads, only rows of the chunk are stored
        __half* dst = static_cast<__half*>(p.out) + (static_cast<size_t>(row0 + r) * H + h) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {
          float v[16];
          tmem_ld16(tl + 256 + c, v);
          tmem_wait_ld();
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const __half2 hv = __floats2half2_rn(v[e] * inv, v[e + 1] * inv);
            w8[e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          if (row_ok) {
            *reinterpret_cast<uint4*>(dst + c) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            *reinterpret_cast<uint4*>(dst + c + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
          }
        }
      }
    } else {
      // ------------------------------------------- normalise z, split into fp16 hi + lo
      uint8_t* zh = sm + L::ZH_OFF;
      uint8_t* zl = sm + L::ZL_OFF;
#pragma unroll 1
      for (int c = 0; c < RQ; c += 32) {
        float v[32];
        if (ok) {
          tmem_ld16(tl + 256 + c, *reinterpret_cast<float(*)[16]>(&v[0]));
          tmem_ld16(tl + 256 + c + 16, *reinterpret_cast<float(*)[16]>(&v[16]));
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0.f;
        }
        uint32_t hw[16], lw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float z0 = v[e] * inv, z1 = v[e + 1] * inv;
          const __half2 hi = __floats2half2_rn(z0, z1);
          const float2 hb = __half22float2(hi);
          const __half2 lo = __floats2half2_rn(z0 - hb.x, z1 - hb.y);
          hw[e / 2] = *reinterpret_cast<const uint32_t*>(&hi);
          lw[e / 2] = *reinterpret_cast<const uint32_t*>(&lo);
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int ch = (c + q4 * 8) / 8;                   // 16-byte chunk index in the row
          const int kb = ch >> 3, cc = ch & 7;
          const int off = kb * 16384 + r * 128 + ((cc ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(zh + off) =
              make_uint4(hw[q4 * 4], hw[q4 * 4 + 1], hw[q4 * 4 + 2], hw[q4 * 4 + 3]);
          *reinterpret_cast<uint4*>(zl + off) =
              make_uint4(lw[q4 * 4], lw[q4 * 4 + 1], lw[q4 * 4 + 2], lw[q4 * 4 + 3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(zq_full);
    }
  }
  __syncwarp();

  // ------------------------------------------------------------------- outputs
  const bool have_o =
      RECON || __all_sync(0xffffffffu, mbar_wait(o_done, 0, abort_flag, p.dev_err));
  tc_fence_after();
  __half* out = static_cast<__half*>(p.out);
  if constexpr (RECON) {
    (void)have_o;
    (void)out;   // written by the softmax warps
  } else if constexpr (NQ == 1) {
    if (warp >= 2 && warp < 6) {
      const int r = (warp & 3) * 32 + lane;
      const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      if (have_o) {   // warp-uniform: every lane loads, only rows of the chunk are stored
        __half* dst = out + (static_cast<size_t>(row0 + r) * H + h) * D;
        const bool store = i0 + r < n;
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {
          float v[16];
          tmem_ld16(tl + c, v);
          tmem_wait_ld();
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const __half2 hv = __floats2half2_rn(v[e], v[e + 1]);
            w8[e / 2] = *reinterpret_cast<const uint32_t*>(&hv);
          }
          if (store) {
            *reinterpret_cast<uint4*>(dst + c) = make_uint4(w8[0], w8[1], w8[2], w8[3]);
            *reinterpret_cast<uint4*>(dst + c + 8) = make_uint4(w8[4], w8[5], w8[6], w8[7]);
          }
        }
      }
    }
  } else {
    constexpr int RPC = L::RPC;
    cluster_sync_all();                 // every slice is done reading its z hi / lo
    float* recv = reinterpret_cast<float*>(sm + L::ZH_OFF);   // [NQ][RPC][D]
    if (warp >= 2 && warp < 6) {
      const int r = (warp & 3) * 32 + lane;
      const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
      const uint32_t dst = map_to_rank(smem_u32(recv), static_cast<uint32_t>(r / RPC)) +
                           ((slice * RPC + r % RPC) * D) * 4;
#pragma unroll 1
      for (int c = 0; c < D; c += 16) {
        float v[16];
        if (have_o) {
          tmem_ld16(tl + c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; e += 4) st_cluster_v4(dst + (c + e) * 4, v[e], v[e + 1], v[e + 2], v[e + 3]);
      }
    }
    cluster_sync_all();
    for (int idx = threadIdx.x; idx < RPC * D / 2; idx += kPfThreads) {
      const int rr = idx / (D / 2), d2 = (idx % (D / 2)) * 2;
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int s = 0; s < NQ; ++s) {
        a0 += recv[(s * RPC + rr) * D + d2];
        a1 += recv[(s * RPC + rr) * D + d2 + 1];
      }
      const int r = slice * RPC + rr;
      if (i0 + r < n)
        *reinterpret_cast<__half2*>(out + (static_cast<size_t>(row0 + r) * H + h) * D + d2) =
            __floats2half2_rn(a0, a1);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// --------------------------------------------------------------------------- launches
template <class S>
cudaError_t prepare_prefill() {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<S, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PfSmem<S, false>::ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_kernel<S, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PfSmem<S, true>::ALLOC);
  return e;
}

// recon: vp is the tensor map of V^ ([rows][H*d], 64 x 128 boxes) and w is not read.
template <class S>
cudaError_t launch_prefill(const CUtensorMap& qhi, const CUtensorMap& qlo, const CUtensorMap& kp,
                           const CUtensorMap& vp, const CUtensorMap& w, const AttnParams& p,
                           int max_tiles, cudaStream_t stream, bool pdl, bool recon) {
  const int NQ = recon ? 1 : PrefillCfg<S>::NQ;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(max_tiles * S::H * NQ);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = recon ? PfSmem<S, true>::ALLOC : PfSmem<S, false>::ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = NQ;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if (recon) return cudaLaunchKernelEx(&cfg, prefill_kernel<S, true>, qhi, qlo, kp, vp, w, p);
  return cudaLaunchKernelEx(&cfg, prefill_kernel<S, false>, qhi, qlo, kp, vp, w, p);
}

template cudaError_t prepare_prefill<ShapeMain>();
template cudaError_t prepare_prefill<ShapeTiny>();
template cudaError_t launch_prefill<ShapeMain>(const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const AttnParams&, int,
                                               cudaStream_t, bool, bool);
template cudaError_t launch_prefill<ShapeTiny>(const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const AttnParams&, int,
                                               cudaStream_t, bool, bool);

}  // namespace rcp
