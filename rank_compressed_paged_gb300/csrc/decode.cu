// Decode attention over low-rank paged coefficients, and the chunked prefill's plan.
//
// A decode call is three launches on the caller's stream (programmatic dependent launch
// between them):
//   A. (gemm.cu)    the rank-space queries q~_h = U_k,h q_h, scaled by log2(e)/sqrt(d) so
//                   the softmax can use exp2, in the same tensor-core launch as a decode
//                   step's append.
//   B. decode_main: persistent split-K kernel.  Every partition plans its own work from
//                   the lengths (no planning launch): the concatenated list of all
//                   requests' blocks is cut into `parts` equal contiguous ranges, one per
//                   CTA.  Per block: tensor-map copies bring the K page (all heads) and the
//                   V page into shared memory; CUDA cores score the block (a warp per 8
//                   heads, 2 heads x 16 tokens per round, one lane per token); an online
//                   softmax with lazy rescaling turns scores into fp16 weights P; one
//                   elected thread issues tcgen05 MMAs Z^T[R x heads] += C_v^T P^T into
//                   tensor memory.  At the end of each (request, range) segment the
//                   accumulator and the running (max, sum) go to a partial record.  The
//                   copies start while launch A still runs: only the compute warps wait
//                   for it (for q~), and the copy thread only before a page that a decode
//                   step's own append writes.  Variants: E4M3 pages (keys scored on the
//                   tensor cores, values widened to fp16 in shared memory by their own
//                   warps), 4-bit pages (key nibbles widened to E4M3 codes first, then the
//                   same), and block-sparse (a page's V is loaded only when some head's
//                   weight in it reaches the threshold; "KV-cache LLM serving" page, "What
//                   it measured", item 3).
//   C. (combine.cu) the split-K combine, merging each request's records in a fixed order
//                   (deterministic), fused with o_h = W_v[:, h*d:(h+1)*d]^T z_h on tensor
//                   cores.
//
// The steps follow the Proxima page: "Per-decode-step attention" (rank-space scoring of
// the compressed cache, split-K with a combine kernel named in "Kernel profiling
// breakdown", plus one matmul per step) and "Per-prefill-chunk attention" (each chunk
// row attends its causal prefix; the plan below lists every chunk row and its tiles).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "launch.h"
#include "ptx.cuh"
#include "quant.cuh"
#include "shape.h"

namespace rcp {

// ----------------------------------------------------------------------------- prefill plan
constexpr int kPlanThreads = 256;
constexpr int kPlanRegRows = 16;

// One CTA: keys attended (qlen) and block-table row (qrow) of every chunk row, the prefix
// sums of their blocks, the list of 128-row query tiles and (reconstructing variant) the
// page prefix sums of the requests with chunk rows.  Launched as a programmatic dependent
// of the kernel before it, which may have produced the lengths, so it waits first.
template <class S>
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const AttnParams p) {
  griddep_wait();
  griddep_launch();
  {
    // ---- plan: qlen / qrow per query row, then cum = prefix sum of ceil(qlen / 16)
    __shared__ int64_t warp_sum[kPlanThreads / 32];
    __shared__ int cu_bad;
    const int tid = threadIdx.x;
    const int32_t max_len = p.bt_stride * kBlockSize;
    if (tid == 0) cu_bad = 0;
    for (int r = tid; r < p.nq; r += kPlanThreads) {
      p.qlen[r] = 0;
      p.qrow[r] = 0;
    }
    __syncthreads();
    // prefill: chunk offsets must not decrease, or two requests could claim the same query
    // rows; if they do, no request is planned (every row stays empty)
    if (p.cu_chunk != nullptr)
      for (int b = tid; b < p.batch; b += kPlanThreads)
        if (p.cu_chunk[b + 1] < p.cu_chunk[b]) cu_bad = 1;
    __syncthreads();
    const bool cu_ok = cu_bad == 0;
    if (!cu_ok && tid == 0) atomicOr(p.dev_err, RCP_DEVERR_BAD_LEN);
    if (p.cu_chunk == nullptr) {
      for (int b = tid; b < p.batch; b += kPlanThreads) {
        const int32_t L = p.seq_lens[b];
        const bool len_ok = L >= 0 && L <= max_len;
        if (!len_ok) atomicOr(p.dev_err, RCP_DEVERR_BAD_LEN);
        p.qlen[b] = len_ok ? L : 0;
        p.qrow[b] = b;
      }
    } else {
      // a warp per request; its lanes write the request's rows
      for (int b = tid >> 5; b < p.batch; b += kPlanThreads / 32) {
        const int32_t L = p.seq_lens[b], c0 = p.cu_chunk[b], c1 = p.cu_chunk[b + 1];
        const int32_t n = c1 - c0;
        if (!cu_ok || L < 0 || L > max_len || c0 < 0 || n < 0 || c1 > p.nq || n > L) {
          if ((tid & 31) == 0) atomicOr(p.dev_err, RCP_DEVERR_BAD_LEN);
          continue;
        }
        for (int32_t i = tid & 31; i < n; i += 32) {
          p.qlen[c0 + i] = L - n + i + 1;   // causal: row i sees keys 0 .. P + i
          p.qrow[c0 + i] = b;
        }
      }
    }
    __syncthreads();
    // block-wide exclusive scan of per-thread sums (contiguous row ranges per thread); a
    // thread's lengths are loaded kPlanRegRows at a time, all loads in flight together
    const int per = (p.nq + kPlanThreads - 1) / kPlanThreads;
    const int r0 = min(p.nq, tid * per), r1 = min(p.nq, r0 + per);
    int64_t s = 0;
    for (int rb = r0; rb < r1; rb += kPlanRegRows) {
      int32_t q[kPlanRegRows];
#pragma unroll
      for (int k = 0; k < kPlanRegRows; ++k) q[k] = rb + k < r1 ? p.qlen[rb + k] : 0;
#pragma unroll
      for (int k = 0; k < kPlanRegRows; ++k) s += (q[k] + kBlockSize - 1) / kBlockSize;
    }
    const int lane = tid & 31, w = tid >> 5;
    int64_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    int64_t acc = incl - s;
    for (int i = 0; i < w; ++i) acc += warp_sum[i];
    if (tid == 0) p.cum[0] = 0;
    for (int rb = r0; rb < r1; rb += kPlanRegRows) {
      int32_t q[kPlanRegRows];
#pragma unroll
      for (int k = 0; k < kPlanRegRows; ++k) q[k] = rb + k < r1 ? p.qlen[rb + k] : 0;
#pragma unroll
      for (int k = 0; k < kPlanRegRows; ++k) {
        acc += (q[k] + kBlockSize - 1) / kBlockSize;
        if (rb + k < r1) p.cum[rb + k + 1] = acc;
      }
    }
    if (p.tile_b != nullptr) {
      // prefill: list the 128-row query tiles of every valid request, in request order
      __syncthreads();
      const int bper = (p.batch + kPlanThreads - 1) / kPlanThreads;
      const int b0 = min(p.batch, tid * bper), b1 = min(p.batch, b0 + bper);
      auto tiles_of = [&](int b) -> int {
        const int32_t L = p.seq_lens[b], c0 = p.cu_chunk[b], c1 = p.cu_chunk[b + 1];
        const int32_t n = c1 - c0;
        const bool ok =
            cu_ok && L >= 0 && L <= max_len && c0 >= 0 && n >= 0 && c1 <= p.nq && n <= L;
        return ok ? (n + 127) / 128 : 0;
      };
      int64_t ts = 0;
      for (int b = b0; b < b1; ++b) ts += tiles_of(b);
      int64_t tin = ts;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, tin, o);
        if (lane >= o) tin += y;
      }
      if (lane == 31) warp_sum[w] = tin;
      __syncthreads();
      int64_t t0 = tin - ts;
      for (int i = 0; i < w; ++i) t0 += warp_sum[i];
      for (int b = b0; b < b1; ++b) {
        const int nt = tiles_of(b);
        for (int i = 0; i < nt; ++i) {
          p.tile_b[t0 + i] = b;
          p.tile_qt[t0 + i] = i;
        }
        t0 += nt;
      }
      if (tid == kPlanThreads - 1) *p.tcount = static_cast<int32_t>(t0);
      if (p.vcum != nullptr) {
        // reconstructing prefill: pages of every request with chunk rows, in request
        // order (the rows of V^)
        __syncthreads();
        int64_t vs = 0;
        for (int b = b0; b < b1; ++b)
          if (tiles_of(b) > 0) vs += (p.seq_lens[b] + kBlockSize - 1) / kBlockSize;
        int64_t vin = vs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int64_t y = __shfl_up_sync(0xffffffffu, vin, o);
          if (lane >= o) vin += y;
        }
        if (lane == 31) warp_sum[w] = vin;
        __syncthreads();
        int64_t v0 = vin - vs;
        for (int i = 0; i < w; ++i) v0 += warp_sum[i];
        if (tid == 0) p.vcum[0] = 0;
        for (int b = b0; b < b1; ++b) {
          if (tiles_of(b) > 0) v0 += (p.seq_lens[b] + kBlockSize - 1) / kBlockSize;
          p.vcum[b + 1] = v0;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------- decode main
constexpr int kAppendSetBits = 9;
constexpr int kAppendSetSize = 1 << kAppendSetBits;   // a step appending more tokens than
                                                      // half this waits before any copy
// FMT: the page format (RCP_PAGES_*).  Quantized pages (F8: E4M3 codes, or 4-bit codes
// with fp16 scales) arrive whole by bulk copies; K pages are scored straight from their
// bytes, V pages land in raw stages and are widened to fp16 in the swizzled layout the
// tensor-core MMA reads (the layout the fp16 path's tensor-map copies produce).
// TSC (E4M3 pages, r_k = 64, heads a multiple of 16): the keys are scored on the tensor
// cores.  Per 8-head group one kind::f8f6f4 MMA (M = 128 key rows of a page, the group's
// heads x 16 tokens; K = r_k) multiplies the E4M3 codes, as the page's TMA copy lands them
// (64-byte swizzle), by the group's query split into four E4M3 terms: head h's q~, scaled
// by a power of two 2^e_h that brings its largest entry into [128, 256), is t0 + t1 + t2
// + t3 with t0 = e4m3(q), t1 = e4m3(q - t0), ... (each residual at most 2^-4 of the one
// before: 2^-16 relative after four terms, down to E4M3's subnormal step).  The 32 columns
// of a group's result are 8 per head pair: (term, head parity); a key row's score is the
// sum of its head's four columns times 2^-e_h.
// 4-bit pages take the same path: the widening warps first write each key page's codes as
// E4M3 values (integers in [-7, 7] are exact in E4M3) in the same 64-byte swizzled layout,
// and a key row's score is further multiplied by the row's scale.
template <class S, int FMT, bool SKIP>
constexpr bool decode_tensor_scores() {
  return (FMT == RCP_PAGES_FP8_E4M3 || (FMT == RCP_PAGES_INT4 && !SKIP)) && S::RK == 64 &&
         S::H % 16 == 0;
}

template <class S, int FMT, bool SKIP = false>
struct DecodeSmem {
  static constexpr bool F8 = FMT != RCP_PAGES_FP16;                 // raw quantized pages
  static constexpr bool TSC = decode_tensor_scores<S, FMT, SKIP>();
  static constexpr bool I4T = TSC && FMT == RCP_PAGES_INT4;         // 4-bit keys widened
  static constexpr int DS = 4;                                      // SKIP: decision ring
  static constexpr int KST = F8 && !TSC ? 3 : 2;                    // key page stages
  static constexpr int VST = 2;                                     // fp16 V stages (MMA A)
  static constexpr int VRS = F8 ? 3 : VST;                          // stages V copies land in
  // P buffers: SKIP keeps four, so the compute warps can run four kept pages ahead of the
  // value MMAs while those pages' values are fetched (a kept page's value copy starts only
  // once the page is decided)
  static constexpr int NPB = SKIP ? 4 : 2;
  static constexpr int KP = FMT == RCP_PAGES_FP8_E4M3 ? S::KPAGE_BYTES / 2   // bytes per K page
                           : FMT == RCP_PAGES_INT4 ? static_cast<int>(Int4Page<S>::KBYTES)
                                                   : S::KPAGE_BYTES;
  static constexpr int VP = FMT == RCP_PAGES_FP8_E4M3 ? S::VPAGE_BYTES / 2   // bytes per V page
                           : FMT == RCP_PAGES_INT4 ? static_cast<int>(Int4Page<S>::VBYTES)
                                                   : S::VPAGE_BYTES;
  // stage strides; I4T: the key stages hold the widened E4M3 operand, the raw 4-bit pages
  // land in KST raw stages of their own
  static constexpr int OPB = S::H * kBlockSize * S::RK;             // E4M3 key operand
  static constexpr int KRPS = (KP + 127) & ~127;
  static constexpr int KPS = I4T ? OPB : KRPS;
  static constexpr int VPS = (VP + 127) & ~127;
  static constexpr int NBAR = 2 * KST + 2 * VRS + 2 * NPB + (F8 ? 2 * VST : 0) + (SKIP ? 2 * DS : 0) +
                              (TSC ? 8 : 0) + (I4T ? 2 * KST : 0);
  static constexpr int P_BYTES = S::HP * 16 * 2;
  static constexpr int V_OFF = 0;                                   // 1024-aligned stages
  static constexpr int K_OFF = V_OFF + VST * S::VSTAGE_BYTES;
  static constexpr int VR_OFF = K_OFF + KST * KPS;                  // raw quantized V stages
  static constexpr int KR_OFF = VR_OFF + (F8 ? VRS * VPS : 0);      // I4T: raw key stages
  static constexpr int P_OFF = KR_OFF + (I4T ? KST * KRPS : 0);
  static constexpr int Q_OFF = P_OFF + NPB * P_BYTES;
  // TSC: the query operand ([H/8 groups][32 rows][r_k] E4M3, K-major without swizzle:
  // 8-row x 16-byte core matrices, 128 bytes apart along K, 512 along the rows; one buffer,
  // rewritten once the previous segment's scoring MMAs completed) and the score factors
  // 2^-e_h per segment parity [2][H]; otherwise q~ in fp32
  static constexpr int QOP_BYTES = (S::H / 8) * 32 * S::RK;
  static constexpr int Q_BYTES = TSC ? QOP_BYTES + 2 * S::H * 4 : S::H * S::RK * 4;
  // I4T: the key-row scales of the page in each score buffer [2][H][16] (fp32)
  static constexpr int KSC_OFF = Q_OFF + Q_BYTES;
  static constexpr int A_OFF = KSC_OFF + (I4T ? 2 * S::H * kBlockSize * 4 : 0);   // alpha[2][HP]
  static constexpr int F_OFF = A_OFF + 2 * S::HP * 4;               // flags[2][4]
  static constexpr int BAR_OFF = F_OFF + 64;                        // NBAR mbarriers
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;               // tmem slot, abort flag
  static constexpr int INFO_OFF = MISC_OFF + 16;                    // valid tokens per stage:
  // K stages, then V; SKIP adds the physical block of each K stage, the decision ring and
  // the info word of each P buffer; TSC the valid tokens of each score buffer; I4T those of
  // each operand stage; SKIP the valid tokens of each decision and (TSC) the physical
  // block of each score buffer
  static constexpr int INFO_BYTES = (2 * KST + VRS + DS + NPB + 2 + KST + DS + 2) * 4;
  // TMEM: the value accumulator [NCHUNK x 128 lanes][HP], then (TSC) two score buffers of
  // H/8 groups x 32 columns
  static constexpr int SCOL = S::NCHUNK * S::HP;
  static constexpr int TMEM_COLS = TSC ? pow2_at_least(SCOL + 2 * (S::H / 8) * 32, 32)
                                       : S::TMEM_COLS;
  // the partition's plan: 32 warp partials of the scans, then the block total, the first
  // request and its first block; then the set of blocks a decode step's append writes
  static constexpr int PLAN_OFF = (INFO_OFF + INFO_BYTES + 7) & ~7;
  static constexpr int HASH_OFF = PLAN_OFF + (32 + 4) * 8;
  // the copy warp's page ring: physical block and valid tokens of two batches of 32 pages
  static constexpr int PG_OFF = HASH_OFF + kAppendSetSize * 4;
  static constexpr int TOTAL = PG_OFF + 2 * 2 * 32 * 4;
  static_assert(PLAN_OFF % 8 == 0 && HASH_OFF % 4 == 0 && A_OFF % 16 == 0 && Q_OFF % 16 == 0 &&
                    BAR_OFF % 8 == 0,
                "region alignment");
  static constexpr int ALLOC = TOTAL + 1024;                        // base alignment slack
  static_assert(KP % 16 == 0 && VP % 16 == 0 && S::VSTAGE_BYTES % 1024 == 0, "alignment");
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(TMEM_COLS <= 512, "tensor memory");
  static_assert(!TSC || (K_OFF % 512 == 0 && KPS % 512 == 0 && Q_OFF % 16 == 0),
                "64-byte swizzled key stages, query operands");
  static_assert(!I4T || (KR_OFF % 16 == 0 && KSC_OFF % 16 == 0), "raw key stages, scales");
};

// Warp 0 copies, warp 1 issues the MMAs, warps 2 .. compute.
// F8: eight compute warps (2-9; scoring E4M3 keys costs more per byte) and warps 10-11,
// which widen the E4M3 V pages while the compute warps score.
// SKIP: warp 0 copies keys only and the last warp copies the value pages the compute warps
// keep.  fp16 pages: eight compute warps (warps 2-9; 10 copies the kept value pages): a
// per-page clock trace showed the four of the dense kernel busy scoring about 3,200 cycles
// of every skipped page while the keys were already resident, so the scoring, not the key
// stream, set the pace (eight: 415 against 443 us at batch 64 x 8192, peaked).  E4M3 pages:
// the tensor-core scoring, with two of the six widening warps building the query operands
// and four widening the kept pages' values.  4-bit pages: the keys are scored on the CUDA
// cores by eight compute warps, and four widening warps widen every kept V page.
// TSC: four compute warps (one per TMEM lane quarter: scores, softmax, weights) and six
// warps that widen the V pages (and build the query operands), so that the widening's
// conversions overlap the softmax's shuffle latencies instead of following them.
template <class S, int FMT, bool SKIP = false>
constexpr int decode_compute_warps() {
  return decode_tensor_scores<S, FMT, SKIP>() ? 4
                                              : ((FMT != RCP_PAGES_FP16 || SKIP) && S::H % 8 == 0) ? 8 : 4;
}
template <class S, int FMT, bool SKIP = false>
constexpr int decode_widen_warps() {
  return decode_tensor_scores<S, FMT, SKIP>()  ? 6
         : FMT == RCP_PAGES_FP16               ? 0
         : (SKIP && S::H % 8 == 0)             ? 4
                                               : 2;
}
template <class S, int FMT, bool SKIP = false>
constexpr int decode_threads() {
  return 32 * (2 + decode_compute_warps<S, FMT, SKIP>() + decode_widen_warps<S, FMT, SKIP>() +
               (SKIP ? 1 : 0));
}

// Two E4M3 codes (low byte first) to an fp16 pair / fp32 pair; E4M3 values are exact in
// fp16.  (Widening by integer bit moves instead measured slower: more instructions.)
__device__ __forceinline__ uint32_t e4m3x2_to_half2_bits(uint16_t codes) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes),
                                                   __NV_E4M3);
  return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t codes) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes),
                                                   __NV_E4M3);
  return __half22float2(__half2(r));
}


// E4M3 pages, an even number of boxes: as widen_v_boxes below, in units of 16 codes (one
// 16-byte load, two 16-byte stores).  A warp's 32 units are 4 tokens x 2 adjacent boxes x 4
// units, so its loads cover four 128-byte row pieces and its stores eight 128-byte stage
// rows: no shared-memory bank is hit twice beyond the minimum.
template <class S, int NT>
__device__ __forceinline__ void widen_v_e4m3_pairs(const uint8_t* src, uint8_t* vb, int nvalid,
                                                   int b0, int b1, int tid) {
  const int n = (b1 - b0) * kBlockSize * 4;
#pragma unroll 2
  for (int idx = tid; idx < n; idx += NT) {
    const int c16 = idx & 3, gl = (idx >> 2) & 1, tl = (idx >> 3) & 3, th = (idx >> 5) & 3;
    const int tt = th * 4 + tl, gb = b0 + (idx >> 7) * 2 + gl;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (tt < nvalid) {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + tt * S::R + gb * 64 + c16 * 16);
      lo.x = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.x & 0xFFFFu));
      lo.y = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.x >> 16));
      lo.z = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.y & 0xFFFFu));
      lo.w = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.y >> 16));
      hi.x = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.z & 0xFFFFu));
      hi.y = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.z >> 16));
      hi.z = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.w & 0xFFFFu));
      hi.w = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.w >> 16));
    }
    uint8_t* row = vb + gb * 2048 + tt * 128;
    *reinterpret_cast<uint4*>(row + (((2 * c16) ^ (tt & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((2 * c16 + 1) ^ (tt & 7)) << 4)) = hi;
  }
}

// 4-bit pages, an even number of boxes: as widen_v_boxes below, in units of 16 codes (8 code
// bytes, one scale), mapped to lanes like widen_v_e4m3_pairs.
template <class S, int NT>
__device__ __forceinline__ void widen_v_int4_pairs(const uint8_t* src, uint8_t* vb, int nvalid,
                                                   int b0, int b1, int tid) {
  const int n = (b1 - b0) * kBlockSize * 4;
  const __half* scales = reinterpret_cast<const __half*>(src + Int4Page<S>::VCODES);
#pragma unroll 8   // measured: 2 -> 652 us, 4 -> 885 us, 8 -> 588 us at batch 64 x 8192
  for (int idx = tid; idx < n; idx += NT) {
    const int c16 = idx & 3, gl = (idx >> 2) & 1, tl = (idx >> 3) & 3, th = (idx >> 5) & 3;
    const int tt = th * 4 + tl, gb = b0 + (idx >> 7) * 2 + gl;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (tt < nvalid) {
      const uint2 raw =
          *reinterpret_cast<const uint2*>(src + tt * (S::R / 2) + gb * 32 + c16 * 8);
      const __half2 sc = __half2half2(scales[tt * (S::R / 64) + gb]);
      lo.x = int4x2_to_half2_bits(raw.x & 0xFFu, sc);
      lo.y = int4x2_to_half2_bits((raw.x >> 8) & 0xFFu, sc);
      lo.z = int4x2_to_half2_bits((raw.x >> 16) & 0xFFu, sc);
      lo.w = int4x2_to_half2_bits(raw.x >> 24, sc);
      hi.x = int4x2_to_half2_bits(raw.y & 0xFFu, sc);
      hi.y = int4x2_to_half2_bits((raw.y >> 8) & 0xFFu, sc);
      hi.z = int4x2_to_half2_bits((raw.y >> 16) & 0xFFu, sc);
      hi.w = int4x2_to_half2_bits(raw.y >> 24, sc);
    }
    uint8_t* row = vb + gb * 2048 + tt * 128;
    *reinterpret_cast<uint4*>(row + (((2 * c16) ^ (tt & 7)) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((2 * c16 + 1) ^ (tt & 7)) << 4)) = hi;
  }
}

// Widens boxes [b0, b1) (64 columns each) of a quantized V page (E4M3: [16][R] codes at src;
// 4-bit: [16][R/2] code bytes then the fp16 scales [16][R/64]) into the fp16 stage vb in
// the layout of the value MMA: box g at g * 2048, token row t at t * 128, 16-byte chunk c
// at chunk c ^ (t % 8).  Tokens at or past nvalid (the sequence end, or a rejected block)
// get zero rows, so whatever those slots hold cannot reach the accumulator through 0 * NaN.
// NT threads, this one is tid.
template <class S, int FMT, int NT>
__device__ __forceinline__ void widen_v_boxes(const uint8_t* src, uint8_t* vb, int nvalid, int b0,
                                              int b1, int tid) {
  if constexpr (FMT == RCP_PAGES_FP8_E4M3 && S::NBOX % 2 == 0) {
    widen_v_e4m3_pairs<S, NT>(src, vb, nvalid, b0, b1, tid);
    return;
  }
  if constexpr (FMT == RCP_PAGES_INT4 && S::NBOX % 2 == 0) {
    widen_v_int4_pairs<S, NT>(src, vb, nvalid, b0, b1, tid);
    return;
  }
  const int n = (b1 - b0) * kBlockSize * 8;
#pragma unroll 4
  for (int idx = tid; idx < n; idx += NT) {
    const int c = idx & 7, tt = (idx >> 3) % kBlockSize, gb = b0 + (idx >> 3) / kBlockSize;
    uint4 o = make_uint4(0, 0, 0, 0);
    if (tt < nvalid) {
      if constexpr (FMT == RCP_PAGES_INT4) {
        // box gb is exactly scale group gb: 8 codes (4 bytes) per 16-byte output chunk
        const uint32_t raw = *reinterpret_cast<const uint32_t*>(src + tt * (S::R / 2) + gb * 32 + c * 4);
        const __half2 sc = __half2half2(reinterpret_cast<const __half*>(
            src + Int4Page<S>::VCODES)[tt * (S::R / 64) + gb]);
        o.x = int4x2_to_half2_bits(raw & 0xFFu, sc);
        o.y = int4x2_to_half2_bits((raw >> 8) & 0xFFu, sc);
        o.z = int4x2_to_half2_bits((raw >> 16) & 0xFFu, sc);
        o.w = int4x2_to_half2_bits(raw >> 24, sc);
      } else {
        const uint2 raw = *reinterpret_cast<const uint2*>(src + tt * S::R + gb * 64 + c * 8);
        o.x = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.x & 0xFFFFu));
        o.y = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.x >> 16));
        o.z = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.y & 0xFFFFu));
        o.w = e4m3x2_to_half2_bits(static_cast<uint16_t>(raw.y >> 16));
      }
    }
    *reinterpret_cast<uint4*>(vb + gb * 2048 + tt * 128 + ((c ^ (tt & 7)) << 4)) = o;
  }
}

__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// Four 4-bit codes (two's complement; code i in nibble i of x's low 16 bits) as four E4M3
// bytes.  A byte permutation looks up the code's low three bits in the table of E4M3 values
// 0..7 and in that of -8..-1; a third, in its sign-replicating mode (selector bit 3 = the
// code's sign bit), marks the negative codes, and the mark picks the second table's byte.
__device__ __forceinline__ uint32_t int4x4_to_e4m3x4(uint32_t x) {
  const uint32_t sel = x & 0x7777u;
  const uint32_t pos = prmt_b32(0x44403800u, 0x4E4C4A48u, sel);   // 0, 1, 2, .. 7
  const uint32_t neg = prmt_b32(0xCACCCED0u, 0xB8C0C4C8u, sel);   // -8, -7, .. -1
  const uint32_t m7 = prmt_b32(0x80808080u, 0x80808080u, x) & 0x7F7F7F7Fu;   // 0x7F: negative
  const uint32_t m = m7 | (m7 << 1);                               // 0xFF: negative
  return (pos & ~m) | (neg & m);
}

// I4T: one 4-bit key page (raw: codes [H][16][r_k / 2] then fp16 scales [H][16]) widened to
// the E4M3 scoring operand op (row r = h * 16 + t, 64 bytes, 16-byte chunk c at c ^ ((r / 2)
// % 4): the layout a 64-byte swizzled tensor copy writes) and its scales to ksc [H][16] fp32.
// NT threads; a unit is 16 code bytes (half a row).
template <class S, int NT>
__device__ __forceinline__ void widen_k_int4(const uint8_t* raw, uint8_t* op, float* ksc,
                                             int tid) {
  static_assert(S::RK == 64, "rows of 32 code bytes");
  constexpr int UNITS = S::H * kBlockSize * 2;
#pragma unroll 8
  for (int u = tid; u < UNITS; u += NT) {
    const int r = u >> 1, half = u & 1;
    const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 32 + half * 16);
    const uint4 lo = make_uint4(int4x4_to_e4m3x4(w.x), int4x4_to_e4m3x4(w.x >> 16),
                                int4x4_to_e4m3x4(w.y), int4x4_to_e4m3x4(w.y >> 16));
    const uint4 hi = make_uint4(int4x4_to_e4m3x4(w.z), int4x4_to_e4m3x4(w.z >> 16),
                                int4x4_to_e4m3x4(w.w), int4x4_to_e4m3x4(w.w >> 16));
    uint8_t* row = op + r * 64;
    const int sw = (r >> 1) & 3;
    *reinterpret_cast<uint4*>(row + (((2 * half) ^ sw) << 4)) = lo;
    *reinterpret_cast<uint4*>(row + (((2 * half + 1) ^ sw) << 4)) = hi;
  }
  const __half* sc = reinterpret_cast<const __half*>(raw + Int4Page<S>::KCODES);
  for (int i = tid; i < S::H * kBlockSize; i += NT) ksc[i] = __half2float(sc[i]);
}

// TSC: the query operand of one request (q: its q~ [H][r_k] fp32) and its score factors
// (qi[h] = 2^-e_h), by 64 threads (vt): two per head, 32 ranks each.  Row n = 8p + 2j + e
// of group g holds term j of head 8g + 2p + e; byte (n, k) of a group sits at
// (n / 8) * 512 + (k / 16) * 128 + (n % 8) * 16 + k % 16.
template <class S>
__device__ __forceinline__ void build_query_operand(const float* q, uint8_t* qo, float* qi,
                                                    int vt) {
  for (int i = vt; i < 2 * S::H; i += 64) {
    const int h = i >> 1, half = i & 1;
    const float4* src = reinterpret_cast<const float4*>(q + h * S::RK + half * 32);
    float x[32];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 v = __ldcg(src + u);
      x[4 * u] = v.x;
      x[4 * u + 1] = v.y;
      x[4 * u + 2] = v.z;
      x[4 * u + 3] = v.w;
    }
    float mx = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) mx = fmaxf(mx, fabsf(x[k]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));   // the partner holds the other half
    int E = 0;
    frexpf(mx, &E);                                         // mx = m 2^E, m in [0.5, 1)
    const int sh = 8 - E;                                   // largest entry -> [128, 256)
    if (half == 0) qi[h] = ldexpf(1.f, -sh);
#pragma unroll
    for (int k = 0; k < 32; ++k) x[k] = ldexpf(x[k], sh);
    uint8_t* base = qo + (h >> 3) * 32 * S::RK + ((h & 7) >> 1) * 512 + (h & 1) * 16 +
                    half * 2 * 128;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[8];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(x[k], __NV_SATFINITE, __NV_E4M3);
        x[k] -= __half2float(__half(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3)));   // exact
        const uint32_t b = static_cast<uint32_t>(c) << (8 * (k & 3));
        w[k >> 2] = (k & 3) ? (w[k >> 2] | b) : b;
      }
      *reinterpret_cast<uint4*>(base + j * 32) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(base + j * 32 + 128) = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
}

constexpr float kRescaleThreshold = 8.f;   // log2 units: weights stay <= 2^8 before a rescale

// Keys of request b: its length when 0 <= L_b <= the table's capacity (max_len), else 0
// (the partition that reports errors sets the length bit for it).
__device__ __forceinline__ int32_t valid_len(int32_t L, int32_t max_len) {
  return (L >= 0 && L <= max_len) ? L : 0;
}

// Walks the requests that a partition's block range crosses; request b covers blocks
// [bstart, bend) of the concatenated list of all requests' blocks.
struct ReqWalker {
  const int32_t* lens;
  int32_t max_len;
  int b;
  int64_t bstart, bend;
  __device__ __forceinline__ int64_t nblk(int r) const {
    return (valid_len(lens[r], max_len) + kBlockSize - 1) / kBlockSize;
  }
  __device__ __forceinline__ void init(const int32_t* l, int32_t ml, int b0, int64_t s0) {
    lens = l;
    max_len = ml;
    b = b0;
    bstart = s0;
    bend = s0 + nblk(b0);
  }
  __device__ __forceinline__ void advance_to(int64_t g) {
    while (g >= bend) {
      ++b;
      bstart = bend;
      bend += nblk(b);
    }
  }
  __device__ __forceinline__ int32_t len() const { return valid_len(lens[b], max_len); }
};

// Blocks a decode step's append writes, as an open-addressing set in shared memory.
__device__ __forceinline__ uint32_t block_hash(int64_t blk) {
  return (static_cast<uint32_t>(blk) * 2654435761u) >> (32 - kAppendSetBits);
}

struct BlockInfo {
  int nvalid;      // tokens of this block that are attended (0 for a rejected block id)
  bool seg_first, seg_last;
};


template <class S, int FMT, bool SKIP>
__global__ void __launch_bounds__(decode_threads<S, FMT, SKIP>(), 1)
    decode_main_kernel(const __grid_constant__ CUtensorMap tmap_v,
                       const __grid_constant__ CUtensorMap tmap_k, const AttnParams p) {
  constexpr bool F8 = FMT != RCP_PAGES_FP16;   // quantized pages (E4M3 or 4-bit)
  // fp16 key pages with 128-byte rows (r_k = 64) arrive 128-byte swizzled (two TMA boxes of
  // 256 rows): chunk c of row r sits at chunk c ^ (r % 8), so the 16 lanes scoring one
  // head read the same logical chunk, conflict-free on the keys and as a broadcast on q~
  constexpr bool KSWZ = !F8 && S::RK == 64;
  using L = DecodeSmem<S, FMT, SKIP>;
  constexpr bool TSC = L::TSC;   // keys scored on the tensor cores (E4M3 or 4-bit pages)
  constexpr bool I4T = L::I4T;   // 4-bit keys widened to E4M3 first
  constexpr int KST = L::KST, VST = L::VST, VRS = L::VRS, HP = S::HP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* vst = sm + L::V_OFF;
  uint8_t* kst = sm + L::K_OFF;
  uint8_t* vraw = sm + L::VR_OFF;
  uint8_t* kraw = sm + L::KR_OFF;                                     // I4T raw key stages
  float* ksc = reinterpret_cast<float*>(sm + L::KSC_OFF);             // I4T [2][H][16]
  uint8_t* pbuf = sm + L::P_OFF;
  float* qs = reinterpret_cast<float*>(sm + L::Q_OFF);
  uint8_t* qop = sm + L::Q_OFF;                                              // TSC [2]
  float* qinv = reinterpret_cast<float*>(sm + L::Q_OFF + L::QOP_BYTES);   // TSC [2][H]
  float* alpha_s = reinterpret_cast<float*>(sm + L::A_OFF);
  int* flags_s = reinterpret_cast<int*>(sm + L::F_OFF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR_OFF);
  uint64_t* kfull = bars;                 // [KST]
  uint64_t* kempty = kfull + KST;         // [KST] the compute warps scored the page
  uint64_t* vfull = kempty + KST;         // [VRS] a V page landed
  uint64_t* vempty = vfull + VRS;         // [VRS] its stage is free (MMA, or F8: widened)
  constexpr int NPB = L::NPB;
  uint64_t* pfull = vempty + VRS;         // [NPB]
  uint64_t* pfree = pfull + NPB;          // [NPB]
  uint64_t* vcvt = pfree + NPB;           // F8 [VST] fp16 V stage written by the widening warps
  uint64_t* vfree = vcvt + VST;           // F8 [VST] fp16 V stage read by its MMAs
  uint64_t* decfull = pfree + NPB + (F8 ? 2 * VST : 0);   // SKIP [DS] a decision was posted
  uint64_t* decempty = decfull + L::DS;                  // SKIP [DS] ... and taken
  uint64_t* sfull = decfull + (SKIP ? 2 * L::DS : 0);    // TSC [2] a page's scores are in TMEM
  uint64_t* sfree = sfull + 2;                           // TSC [2] ... and were read
  uint64_t* qfull = sfree + 2;                           // TSC [2] a segment's query operand
  uint64_t* qfree = qfull + 2;                           // TSC [2] ... its MMAs completed
  uint64_t* kopfull = qfree + 2;                         // I4T [KST] widened key operand
  uint64_t* kopempty = kopfull + KST;                    // I4T [KST] ... its MMAs completed
  constexpr int NTHR = decode_threads<S, FMT, SKIP>();
  constexpr int NCW = decode_compute_warps<S, FMT, SKIP>();   // compute warps 2 .. NCW+1
  // F8: V boxes widened by warps 10-11; the compute warps widen the remaining ones (a
  // split measured to balance the two groups' time per block)
  constexpr int NWW = decode_widen_warps<S, FMT, SKIP>();   // widening warps NCW+2 ..
  // warps that widen V pages: all widening warps, but with tensor-core scoring and
  // skipping the first two build the query operands only (they follow every page, the
  // others the kept pages)
  constexpr int NVW = (TSC && SKIP) ? NWW - 2 : NWW;
  // (4-bit pages: the widening warps also widen the key codes, so the compute warps take
  // 10 of the 16 value boxes: measured 521 us at batch 64 x 8192 against 588 us for none)
  // (SKIP: all of them, in the order of the kept pages)
  constexpr int WB =
      (SKIP || (TSC && FMT == RCP_PAGES_FP8_E4M3)) ? S::NBOX : S::NBOX >= 16 ? 6 : S::NBOX;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC_OFF + 4);
  // tokens of the block in each stage that are attended, published by the copy thread
  // before it arms the stage's barrier (so a waiter sees it), so that no other warp
  // reads the block table or lengths from global memory on its critical path
  int* kinfo = reinterpret_cast<int*>(sm + L::INFO_OFF);
  int* vinfo = kinfo + KST;
  // SKIP: the physical block of each K stage; the decision ring (physical block of each
  // kept page, in order, -1 = no more pages); per P buffer 1 = first page of a segment,
  // 0 = a later one, -1 = no more pages
  int* kphys = vinfo + VRS;
  int* dec_s = kphys + KST;
  int* pinfo = dec_s + L::DS;
  int* sinfo = pinfo + NPB; // TSC: valid tokens of the page in each score buffer
  int* oinfo = sinfo + 2;   // I4T: valid tokens of the page in each operand stage
  int* dec_n = oinfo + KST; // SKIP: valid tokens of each kept page of the decision ring
  int* sphys = dec_n + L::DS;   // SKIP + TSC: physical block of the page in each score buffer

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  // prologue: nothing here reads what the previous kernel writes
  if (threadIdx.x == 0) {
    for (int i = 0; i < KST; ++i) {
      mbar_init(&kfull[i], 1);
      // TSC: the scoring MMAs' commit; I4T: the widening warps (raw stage)
      mbar_init(&kempty[i], I4T ? NWW : TSC ? 1 : NCW);
      if constexpr (I4T) {
        mbar_init(&kopfull[i], NWW);
        mbar_init(&kopempty[i], 1);
      }
    }
    if constexpr (TSC) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&sfull[i], 2);    // the MMA thread's arrive (after sinfo) + the commit
        mbar_init(&sfree[i], NCW);
        mbar_init(&qfull[i], 2);    // the two widening warps
        mbar_init(&qfree[i], 1 + NCW);   // the MMAs' commit + each compute warp's read of
                                         // the score factors
      }
    }
    for (int i = 0; i < VRS; ++i) {
      mbar_init(&vfull[i], 1);
      mbar_init(&vempty[i], F8 ? NVW + (WB < S::NBOX ? NCW : 0) : 1);
    }
    if constexpr (F8) {
      for (int i = 0; i < VST; ++i) {
        mbar_init(&vcvt[i], NVW);
        mbar_init(&vfree[i], 1);
      }
    }
    for (int i = 0; i < NPB; ++i) {
      mbar_init(&pfull[i], NCW);
      mbar_init(&pfree[i], 1);
    }
    if constexpr (SKIP) {
      for (int i = 0; i < L::DS; ++i) {
        mbar_init(&decfull[i], 1);
        mbar_init(&decempty[i], 1);
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  // Zero both P buffers (padded head rows stay zero) and any part of a V stage that no
  // copy fills (value rank below a multiple of 128: those MMA rows are never stored).
  for (int i = threadIdx.x; i < NPB * L::P_BYTES / 16; i += NTHR)
    reinterpret_cast<uint4*>(pbuf)[i] = make_uint4(0, 0, 0, 0);
  if constexpr (S::NBOX < 2 * S::NCHUNK) {
    constexpr int ZB = (2 * S::NCHUNK - S::NBOX) * 2048 / 16;
    for (int s = 0; s < VST; ++s)
      for (int i = threadIdx.x; i < ZB; i += NTHR)
        reinterpret_cast<uint4*>(vst + s * S::VSTAGE_BYTES + S::NBOX * 2048)[i] =
            make_uint4(0, 0, 0, 0);
  }

  // ---- plan, from the lengths alone (inputs of the call, complete before the launch
  // ahead of this one started, so they are read before waiting on it): request b covers
  // ceil(L_b / 16) blocks of the concatenated list (none for an invalid length); the list
  // is cut into G equal ranges, one per partition.  Partition 0 also reports invalid
  // lengths and writes the block prefix sums for the combine.
  constexpr int NWARP = NTHR / 32;
  const int32_t max_len = p.bt_stride * kBlockSize;
  int64_t* red = reinterpret_cast<int64_t*>(sm + L::PLAN_OFF);   // [32] warp partials
  int64_t* plan = red + 32;                                       // first request, its block
  {
    int64_t part = 0;
    for (int b = threadIdx.x; b < p.nq; b += NTHR)
      part += (valid_len(p.seq_lens[b], max_len) + kBlockSize - 1) / kBlockSize;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) red[warp] = part;
    if (threadIdx.x == 0) {
      plan[0] = -1;
      plan[1] = 0;
    }
  }
  __syncthreads();
  int64_t T = 0;
#pragma unroll
  for (int i = 0; i < NWARP; ++i) T += red[i];
  // never more partitions than blocks, so every partition's range is non-empty, and at
  // least decode_min_pages(nq) blocks per partition, so that small batches do not spread
  // over more partitions than pays for their split-K records (128 KiB each)
  const int64_t Gm = (T + decode_min_pages<S>(p.nq) - 1) / decode_min_pages<S>(p.nq);
  const int G = static_cast<int>(Gm < gridDim.x ? Gm : gridDim.x);
  const bool active = cta < G;   // uniform over the CTA
  const int64_t g0 = active ? static_cast<int64_t>(cta) * T / G : 0;
  const int64_t g1 = active ? static_cast<int64_t>(cta + 1) * T / G : 0;
  const bool writer = cta == 0;
  __syncthreads();   // every thread has its total before red[] is reused
  if (writer) {
    if (threadIdx.x == 0) p.cum[0] = 0;
    // the combine's arrival counters, one per (tile of requests, head)
    const int groups = (p.nq + CombineCfg<S>::NT - 1) / CombineCfg<S>::NT * S::H;
    for (int i = threadIdx.x; i < groups; i += NTHR) p.ucnt[i] = 0;
  }
  if (writer || active) {
    // chunked block-wide scan of the block counts until the request holding g0 is found
    // (partition 0 scans them all)
    int64_t base = 0;
    for (int c0 = 0; c0 < p.nq; c0 += NTHR) {
      const int b = c0 + threadIdx.x;
      int64_t v = 0;
      if (b < p.nq) {
        const int32_t Lb = p.seq_lens[b];
        if (writer && (Lb < 0 || Lb > max_len)) atomicOr(p.dev_err, RCP_DEVERR_BAD_LEN);
        v = (valid_len(Lb, max_len) + kBlockSize - 1) / kBlockSize;
      }
      int64_t incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) red[warp] = incl;
      __syncthreads();
      int64_t tot = 0;
#pragma unroll
      for (int i = 0; i < NWARP; ++i) {
        if (i < warp) incl += red[i];
        tot += red[i];
      }
      incl += base;
      if (b < p.nq) {
        if (writer) p.cum[b + 1] = incl;
        if (active && v > 0 && incl - v <= g0 && g0 < incl) {
          plan[0] = b;
          plan[1] = incl - v;
        }
      }
      base += tot;
      __syncthreads();   // red[] is reused; plan[] is visible
      if (!writer && plan[0] >= 0) break;   // uniform: read after the barrier
    }
  }
  const int b_first = static_cast<int>(plan[0]);
  const int64_t s_first = plan[1];
  // ---- a decode step's own append (the launch ahead) writes these blocks: the copy thread
  // waits for it before copying one of them, and before any copy when the step appends
  // more tokens than the set holds
  int* aset = reinterpret_cast<int*>(sm + L::HASH_OFF);
  const bool step = p.n_slots > 0;
  const bool wait_first = p.n_slots > kAppendSetSize / 2;
  if (step && !wait_first) {
    for (int i = threadIdx.x; i < kAppendSetSize; i += NTHR) aset[i] = -1;
    __syncthreads();
    for (int i = threadIdx.x; i < p.n_slots; i += NTHR) {
      const int64_t sl = p.slots[i];
      if (sl < 0 || sl >= p.num_blocks * kBlockSize) continue;
      const int blk = static_cast<int>(sl / kBlockSize);
      uint32_t h = block_hash(blk);
      for (int probe = 0; probe < kAppendSetSize; ++probe) {
        const int prev = atomicCAS(&aset[h], -1, blk);
        if (prev == -1 || prev == blk) break;
        h = (h + 1) & (kAppendSetSize - 1);
      }
    }
  }
  auto appended = [&](int64_t blk) {
    uint32_t h = block_hash(blk);
    for (int probe = 0; probe < kAppendSetSize; ++probe) {
      const int v = aset[h];
      if (v == blk) return true;
      if (v < 0) return false;
      h = (h + 1) & (kAppendSetSize - 1);
    }
    return false;
  };

  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap_v);
  griddep_launch();   // the combine + up-projection may start its prologue

  ReqWalker walk;
  if (active) walk.init(p.seq_lens, max_len, b_first, s_first);

  if (!active) {
    // no blocks for this CTA
  } else if (warp == 0) {
    // ------------------------------------------------------------------ copy producer
    // The whole warp looks up the block ids and valid tokens of 32 pages at a time (lane l:
    // page c0 + l), one batch ahead of the copies, so that lane 0 never waits on a table
    // load; lane 0 issues the copies.
    int* pg_phys = reinterpret_cast<int*>(sm + L::PG_OFF);   // [2][32]
    int* pg_nval = pg_phys + 64;                              // [2][32]
    ReqWalker lw = walk;
    auto lookup = [&](int64_t gb, int& ph, int& nv) {
      const int64_t g = gb + lane;
      ph = 0;
      nv = 0;
      if (g < g1) {
        lw.advance_to(g);
        const int64_t j = g - lw.bstart;
        const int64_t raw = p.block_table[static_cast<int64_t>(lw.b) * p.bt_stride + j];
        const bool bad = raw < 0 || raw >= p.num_blocks;
        if (bad) atomicOr(p.dev_err, RCP_DEVERR_BAD_BLOCK);
        ph = bad ? 0 : static_cast<int>(raw);
        const int64_t left = lw.len() - j * kBlockSize;
        nv = bad ? 0 : static_cast<int>(left < kBlockSize ? left : kBlockSize);
      }
    };
    {
      int ph, nv;
      lookup(g0, ph, nv);
      pg_phys[lane] = ph;
      pg_nval[lane] = nv;
    }
    __syncwarp();
    const uint64_t pol = policy_evict_first();
    const uint8_t* kpages = static_cast<const uint8_t*>(p.k_pages);
    int64_t nk = 0, nv = 0;
    bool waited = !step;
    bool stop = false;
    for (int64_t c0 = g0, batch = 0; c0 < g1 && !stop; c0 += 32, ++batch) {
      int ph_n = 0, nv_n = 0;   // the next batch: loads in flight while lane 0 copies
      if (c0 + 32 < g1) lookup(c0 + 32, ph_n, nv_n);
      if (lane == 0) {
        const int cnt = static_cast<int>(g1 - c0 < 32 ? g1 - c0 : 32);
        for (int i = 0; i < cnt; ++i) {
          const int64_t it = c0 - g0 + i;
          const int64_t phys = pg_phys[(batch & 1) * 32 + i];
          const int nvalid = pg_nval[(batch & 1) * 32 + i];
          if (!waited && (wait_first || appended(phys))) {
            griddep_wait();   // the step's append has written this block
            waited = true;
          }
          const int ks = static_cast<int>(it % KST);
          if (it >= KST && !mbar_wait(&kempty[ks], ((it / KST) - 1) & 1, abort_flag, p.dev_err)) {
            stop = true;
            break;
          }
          kinfo[ks] = nvalid;
          if constexpr (SKIP) kphys[ks] = static_cast<int>(phys);
          mbar_arrive_expect_tx(&kfull[ks], L::KP);
          if constexpr (KSWZ || (TSC && !I4T)) {
            constexpr int ROWS = S::H * kBlockSize;   // key rows of a page
            constexpr int RB = TSC ? S::RK : S::RK * 2;   // bytes per row
#pragma unroll
            for (int half = 0; half < ROWS / 256; ++half)
              tma_load_2d_hint(kst + ks * L::KPS + half * 256 * RB, &tmap_k, 0,
                               static_cast<int32_t>(phys * ROWS + half * 256), &kfull[ks], pol);
          } else {
            bulk_g2s_hint(I4T ? kraw + ks * L::KRPS : kst + ks * L::KPS, kpages + phys * L::KP,
                          L::KP, &kfull[ks], pol);
          }
          ++nk;
          if constexpr (SKIP) continue;   // values wait until the page is known to be needed
          const int vs = static_cast<int>(it % VRS);
          if (it >= VRS && !mbar_wait(&vempty[vs], ((it / VRS) - 1) & 1, abort_flag, p.dev_err)) {
            stop = true;
            break;
          }
          vinfo[vs] = nvalid;
          mbar_arrive_expect_tx(&vfull[vs], L::VP);
          if constexpr (F8) {
            // the page's [16][R] codes, contiguous
            bulk_g2s_hint(vraw + vs * L::VPS,
                          static_cast<const uint8_t*>(p.v_pages) + phys * L::VP, L::VP,
                          &vfull[vs], pol);
          } else {
#pragma unroll 1
            for (int bx = 0; bx < S::NBOX; ++bx)
              tma_load_2d_hint(vst + vs * S::VSTAGE_BYTES + bx * 2048, &tmap_v, bx * 64,
                               static_cast<int32_t>(phys * kBlockSize), &vfull[vs], pol);
          }
          ++nv;
        }
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      __syncwarp();   // lane 0 has read this batch's slot before it is rewritten
      pg_phys[((batch + 1) & 1) * 32 + lane] = ph_n;
      pg_nval[((batch + 1) & 1) * 32 + lane] = nv_n;
      __syncwarp();
    }
    if (lane == 0 && *abort_flag) {   // let copies already in flight land before the CTA exits
      for (int64_t i = (nk > KST ? nk - KST : 0); i < nk; ++i)
        mbar_wait_drain(&kfull[i % KST], (i / KST) & 1);
      for (int64_t i = (nv > VRS ? nv - VRS : 0); i < nv; ++i)
        mbar_wait_drain(&vfull[i % VRS], (i / VRS) & 1);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_f16(128, HP, /*a_mn_major=*/true, /*b_mn_major=*/false);
      int64_t issued = 0;
      if constexpr (SKIP && !TSC) {
        // kept pages only, in order; the info word of each P buffer says whether the page
        // opens a segment (accumulator overwritten) or that no page follows
        for (int64_t kk = 0;; ++kk) {
          const int vs = static_cast<int>(kk % VST), ps = static_cast<int>(kk % NPB);
          if (!mbar_wait(&pfull[ps], (kk / NPB) & 1, abort_flag, p.dev_err)) break;
          const int info = pinfo[ps];
          if (info < 0) break;
          if (!mbar_wait(F8 ? &vcvt[vs] : &vfull[vs], (kk / VST) & 1, abort_flag, p.dev_err)) break;
          tc_fence_after();
          const uint32_t vaddr = smem_u32(vst + vs * S::VSTAGE_BYTES);
          const uint64_t bdesc = make_sdesc(smem_u32(pbuf + ps * L::P_BYTES), 128, 256, kSwizzleNone);
#pragma unroll
          for (int i = 0; i < S::NCHUNK; ++i) {
            const uint64_t adesc = make_sdesc(vaddr + i * 4096, 2048, 1024, kSwizzle128B);
            umma_f16(tmem_base + i * HP, adesc, bdesc, idesc, info ? 0u : 1u);
          }
          umma_commit(F8 ? &vfree[vs] : &vempty[vs]);
          umma_commit(&pfree[ps]);
          ++issued;
        }
      }
      // TSC: the scores of page it + 1 go out before the values of page it, so that the
      // compute warps find the next page's scores ready when they finish this one
      ReqWalker wsc = walk;   // the scoring MMAs' own walk, one page ahead
      int64_t nseg = 0;       // segments whose scoring has started
      auto issue_scores = [&](int64_t g, int64_t it) -> bool {
        wsc.advance_to(g);
        const bool first = (g == g0) || (g == wsc.bstart);
        const bool last = (g == g1 - 1) || (g + 1 == wsc.bend);
        if (first) ++nseg;
        const int qb = static_cast<int>((nseg - 1) & 1);
        const int ks = static_cast<int>(it % KST), sb = static_cast<int>(it & 1);
        if (first && !mbar_wait(&qfull[qb], ((nseg - 1) >> 1) & 1, abort_flag, p.dev_err))
          return false;
        if (!mbar_wait(I4T ? &kopfull[ks] : &kfull[ks], (it / KST) & 1, abort_flag, p.dev_err))
          return false;
        if (it >= 2 && !mbar_wait(&sfree[sb], ((it >> 1) - 1) & 1, abort_flag, p.dev_err))
          return false;
        sinfo[sb] = I4T ? oinfo[ks] : kinfo[ks];
        mbar_arrive(&sfull[sb]);
        tc_fence_after();
        constexpr uint32_t idesc_s = make_idesc_f16(128, 32, false, false);   // E4M3 = format 0
        const uint32_t kaddr = smem_u32(kst + ks * L::KPS);
        const uint32_t qaddr = smem_u32(qop);
#pragma unroll
        for (int gi = 0; gi < S::H / 8; ++gi) {
#pragma unroll
          for (int kk = 0; kk < S::RK / 32; ++kk) {
            const uint64_t adesc =
                make_sdesc(kaddr + gi * 128 * S::RK + kk * 32, 16, 512, kSwizzle64B);
            const uint64_t bdesc =
                make_sdesc(qaddr + gi * 32 * S::RK + kk * 256, 128, 512, kSwizzleNone);
            umma_f8(tmem_base + L::SCOL + sb * (S::H / 8) * 32 + gi * 32, adesc, bdesc, idesc_s,
                    kk > 0 ? 1u : 0u);
          }
        }
        umma_commit(&sfull[sb]);
        umma_commit(I4T ? &kopempty[ks] : &kempty[ks]);
        if (last) umma_commit(&qfree[qb]);
        return true;
      };
      if constexpr (SKIP && TSC) {
        // the scores of every page and the values of the kept pages, each issued as soon as
        // it is ready (non-blocking probes): a page's scores never wait for an earlier
        // page's decision, so the compute warps always find the next scores in flight
        int64_t it_s = 0, kk = 0;   // pages scored, kept pages accumulated
        uint64_t t_idle = 0;
        while (true) {
          bool progress = false;
          if (g0 + it_s < g1) {
            const int64_t g = g0 + it_s;
            wsc.advance_to(g);
            const bool first = (g == g0) || (g == wsc.bstart);
            const int ks = static_cast<int>(it_s % KST), sb = static_cast<int>(it_s & 1);
            const bool ready =
                (!first || mbar_test_wait(&qfull[nseg & 1], (nseg >> 1) & 1)) &&
                mbar_test_wait(&kfull[ks], (it_s / KST) & 1) &&
                (it_s < 2 || mbar_test_wait(&sfree[sb], ((it_s >> 1) - 1) & 1));
            if (ready) {
              sphys[sb] = kphys[ks];
              issue_scores(g, it_s);   // its waits are satisfied: they return at once
              ++it_s;
              progress = true;
            }
          }
          const int ps = static_cast<int>(kk % NPB), vs = static_cast<int>(kk % VST);
          if (mbar_test_wait(&pfull[ps], (kk / NPB) & 1)) {
            const int info = pinfo[ps];
            if (info < 0) break;   // every page is decided and every kept page accumulated
            if (mbar_test_wait(&vcvt[vs], (kk / VST) & 1)) {
              tc_fence_after();
              const uint32_t vaddr = smem_u32(vst + vs * S::VSTAGE_BYTES);
              const uint64_t bdesc =
                  make_sdesc(smem_u32(pbuf + ps * L::P_BYTES), 128, 256, kSwizzleNone);
#pragma unroll
              for (int i = 0; i < S::NCHUNK; ++i) {
                const uint64_t adesc = make_sdesc(vaddr + i * 4096, 2048, 1024, kSwizzle128B);
                umma_f16(tmem_base + i * HP, adesc, bdesc, idesc, info ? 0u : 1u);
              }
              umma_commit(&vfree[vs]);
              umma_commit(&pfree[ps]);
              ++kk;
              ++issued;
              progress = true;
            }
          }
          if (progress) {
            t_idle = 0;
            continue;
          }
          if (*abort_flag) break;
          if (t_idle == 0) {
            t_idle = globaltimer_ns();
          } else if (globaltimer_ns() - t_idle > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(p.dev_err, RCP_DEVERR_TIMEOUT);
            break;
          }
        }
      }
      bool run = true;
      if constexpr (TSC && !SKIP) run = g0 < g1 && issue_scores(g0, 0);
      for (int64_t g = g0, it = 0; !SKIP && run && g < g1; ++g, ++it) {
        if constexpr (TSC)
          if (g + 1 < g1 && !issue_scores(g + 1, it + 1)) break;
        walk.advance_to(g);
        const bool seg_first = (g == g0) || (g == walk.bstart);
        const int vs = static_cast<int>(it % VST), ps = static_cast<int>(it & 1);
        if (!mbar_wait(F8 ? &vcvt[vs] : &vfull[vs], (it / VST) & 1, abort_flag, p.dev_err)) break;
        if (!mbar_wait(&pfull[ps], (it >> 1) & 1, abort_flag, p.dev_err)) break;
        tc_fence_after();
        const uint32_t vaddr = smem_u32(vst + vs * S::VSTAGE_BYTES);
        const uint64_t bdesc = make_sdesc(smem_u32(pbuf + ps * L::P_BYTES), 128, 256, kSwizzleNone);
#pragma unroll
        for (int i = 0; i < S::NCHUNK; ++i) {
          const uint64_t adesc = make_sdesc(vaddr + i * 4096, 2048, 1024, kSwizzle128B);
          umma_f16(tmem_base + i * HP, adesc, bdesc, idesc, seg_first ? 0u : 1u);
        }
        umma_commit(F8 ? &vfree[vs] : &vempty[vs]);
        umma_commit(&pfree[ps]);
        ++issued;
      }
      if (issued > 0) mbar_wait_drain(&pfree[(issued - 1) % NPB], ((issued - 1) / NPB) & 1);
    }
  } else if (SKIP && warp == 2 + NCW + NWW) {
    // ------------------------------------------ SKIP: value pages of the kept pages
    // (F8: the raw pages, into the stages the widening warps read; after the last one a
    // stage whose info word is -1 tells them that no page follows)
    if (lane == 0) {
      if (step) griddep_wait();   // pages an append ahead of this launch wrote
      const uint64_t pol = policy_evict_first();
      constexpr int NS = F8 ? VRS : VST;   // stages the copies land in
      int64_t nv = 0;
      for (int64_t n = 0;; ++n) {
        const int ds = static_cast<int>(n % L::DS);
        if (!mbar_wait(&decfull[ds], (n / L::DS) & 1, abort_flag, p.dev_err)) break;
        const int phys = dec_s[ds], nval = dec_n[ds];
        mbar_arrive(&decempty[ds]);
        const int vs = static_cast<int>(nv % NS);
        if (phys < 0 && !F8) break;
        if (nv >= NS && !mbar_wait(&vempty[vs], ((nv / NS) - 1) & 1, abort_flag, p.dev_err)) break;
        if constexpr (F8) {
          vinfo[vs] = phys < 0 ? -1 : nval;
          if (phys < 0) {
            mbar_arrive(&vfull[vs]);
            break;
          }
          mbar_arrive_expect_tx(&vfull[vs], L::VP);
          bulk_g2s_hint(vraw + vs * L::VPS,
                        static_cast<const uint8_t*>(p.v_pages) + static_cast<int64_t>(phys) * L::VP,
                        L::VP, &vfull[vs], pol);
        } else {
          mbar_arrive_expect_tx(&vfull[vs], L::VP);
#pragma unroll 1
          for (int bx = 0; bx < S::NBOX; ++bx)
            tma_load_2d_hint(vst + vs * S::VSTAGE_BYTES + bx * 2048, &tmap_v, bx * 64,
                             phys * kBlockSize, &vfull[vs], pol);
        }
        ++nv;
      }
      if (*abort_flag)   // let copies already in flight land before the CTA exits
        for (int64_t i = (nv > NS ? nv - NS : 0); i < nv; ++i)
          mbar_wait_drain(&vfull[i % NS], (i / NS) & 1);
    }
  } else if (F8 && warp >= 2 + NCW) {
    // ------------------------------------------ F8: widen E4M3 V pages to fp16 stages
    // boxes [0, WB) here; the compute warps widen the rest after writing P
    const int vt = threadIdx.x - 32 * (2 + NCW);   // 0 .. 32 NWW - 1
    const bool q_builder = vt < 64;                  // TSC: warps NCW+2, NCW+3
    ReqWalker wq = walk;   // TSC: these warps also write each segment's query operand
    int64_t nseg = 0;
    bool q_ready = false;
    // SKIP: the kept pages, in order, until a stage whose info word is -1
    // (TSC: the query builders take no part; the other widening warps do the values)
    const bool v_widener = !(TSC && SKIP) || !q_builder;
    const int vw = (TSC && SKIP) ? vt - 64 : vt;   // 0 .. 32 NVW - 1 over the value wideners
    for (int64_t n = 0; SKIP && v_widener; ++n) {
      const int vr = static_cast<int>(n % VRS), vs = static_cast<int>(n % VST);
      bool ok = mbar_wait(&vfull[vr], (n / VRS) & 1, abort_flag, p.dev_err);
      if (n >= VST) ok = mbar_wait(&vfree[vs], ((n / VST) - 1) & 1, abort_flag, p.dev_err) && ok;
      if (!__all_sync(0xffffffffu, ok)) break;
      const int nval = vinfo[vr];
      if (nval < 0) break;
      widen_v_boxes<S, FMT, 32 * NVW>(vraw + vr * L::VPS, vst + vs * S::VSTAGE_BYTES, nval, 0, WB, vw);
      fence_proxy_async_smem();   // generic stores -> the MMA's async-proxy reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&vempty[vr]);   // this warp is done with the raw page
        mbar_arrive(&vcvt[vs]);     // its part of the fp16 stage is ready
      }
    }
    // every page in order: the query operands at segment starts (TSC), the 4-bit key codes
    // (I4T) and, without skipping, the V pages
    for (int64_t g = g0, it = 0; (!SKIP || (TSC && q_builder)) && g < g1; ++g, ++it) {
      if constexpr (TSC) {
        wq.advance_to(g);
        if (q_builder && (g == g0 || g == wq.bstart)) {
          ++nseg;
          const int qb = static_cast<int>((nseg - 1) & 1);
          // the previous segment's scoring MMAs have read the operand, and the compute
          // warps hold its score factors (qfree of segment nseg - 2)
          const int64_t prev = nseg - 2;
          bool ok = prev < 0 ||
                    mbar_wait(&qfree[prev & 1], (prev >> 1) & 1, abort_flag, p.dev_err);
          if (!__all_sync(0xffffffffu, ok)) break;
          if (!q_ready) {
            griddep_wait();   // the rank-space queries of the launch ahead are written
            q_ready = true;
          }
          build_query_operand<S>(p.qt + static_cast<size_t>(wq.b) * S::H * S::RK, qop,
                                 qinv + qb * S::H, vt);
          fence_proxy_async_smem();   // generic stores -> the MMA's async-proxy reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&qfull[qb]);
        }
      }
      if constexpr (SKIP) continue;   // the values of kept pages are the other warps' part
      if constexpr (I4T) {
        // this page's key codes as the E4M3 scoring operand, once the raw page landed, the
        // operand stage's MMAs completed and the compute warps read the scales two pages ago
        const int ks = static_cast<int>(it % KST), sb = static_cast<int>(it & 1);
        bool kok = mbar_wait(&kfull[ks], (it / KST) & 1, abort_flag, p.dev_err);
        if (it >= KST)
          kok = mbar_wait(&kopempty[ks], ((it / KST) - 1) & 1, abort_flag, p.dev_err) && kok;
        if (it >= 2) kok = mbar_wait(&sfree[sb], ((it >> 1) - 1) & 1, abort_flag, p.dev_err) && kok;
        if (!__all_sync(0xffffffffu, kok)) break;
        widen_k_int4<S, 32 * NWW>(kraw + ks * L::KRPS, kst + ks * L::KPS,
                                  ksc + sb * S::H * kBlockSize, vt);
        if (vt == 0) oinfo[ks] = kinfo[ks];
        fence_proxy_async_smem();   // generic stores -> the MMA's async-proxy reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&kempty[ks]);    // the raw page may be overwritten
          mbar_arrive(&kopfull[ks]);   // the operand is ready
        }
      }
      const int vr = static_cast<int>(it % VRS), vs = static_cast<int>(it % VST);
      bool ok = mbar_wait(&vfull[vr], (it / VRS) & 1, abort_flag, p.dev_err);
      if (it >= VST) ok = mbar_wait(&vfree[vs], ((it / VST) - 1) & 1, abort_flag, p.dev_err) && ok;
      if (!__all_sync(0xffffffffu, ok)) break;
      widen_v_boxes<S, FMT, 32 * NWW>(vraw + vr * L::VPS, vst + vs * S::VSTAGE_BYTES, vinfo[vr], 0,
                                      WB, vt);
      fence_proxy_async_smem();   // generic stores -> the MMA's async-proxy reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&vempty[vr]);   // this warp is done with the raw page
        mbar_arrive(&vcvt[vs]);     // its part of the fp16 stage is ready
      }
    }
  } else {
    // ------------------------------------------------- scores, softmax, P, epilogue
    constexpr int HPW = S::H / NCW;             // heads per compute warp
    constexpr int ROUNDS = (HPW + 1) / 2;       // two heads (16 lanes each) per round
    constexpr int NCH = S::RK / 8;              // 16-byte chunks per K row
    const int cw = warp - 2;                    // head group
    const int quarter = warp & 3;               // TMEM lane quarter this warp may access
    const int hl = lane >> 4, t = lane & 15;
    const int ctid = threadIdx.x - 64;          // 0 .. 32*NCW-1 over the compute warps
    constexpr int CT = 32 * NCW;                // compute threads
    // warps sharing a TMEM lane quarter split the accumulator's 128-row chunks
    const int chunk0 = cw / 4;
    constexpr int CSTEP = NCW / 4;
    float m_run[ROUNDS], l_run[ROUNDS];
    float mt[ROUNDS];   // SKIP: largest score of the segment's kept pages (log2 units)
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) { m_run[r] = -INFINITY; l_run[r] = 0.f; mt[r] = -INFINITY; }
    const float4* qs4 = reinterpret_cast<const float4*>(qs);
    // warp cw takes heads cw*HPW .., two per round (one per half-warp)
    auto head_ok = [&](int r) { return 2 * r + hl < HPW; };
    // TSC: a warp reads the score rows of its TMEM lane quarter: heads 8 gi + 2 quarter +
    // (0, 1) of groups gi = (cw / 4) ROUNDS + r
    auto head_of = [&](int r) {
      return TSC ? 8 * ((cw / 4) * ROUNDS + r) + 2 * quarter + hl : cw * HPW + 2 * r + hl;
    };
    static_assert(!TSC || S::H == 8 * ROUNDS * (NCW / 4), "tensor scoring head split");
    float qf[ROUNDS];   // TSC: the segment's score factors 2^-e_h of this lane's heads
    int64_t nseg_c = 0;
    int64_t kk = 0;     // pages accumulated so far (SKIP: the kept ones), orders P / V use
    int64_t nd = 0;     // SKIP: decisions posted to the value-copy warp
    bool aborted = false;
    griddep_wait();     // the rank-space queries of the launch ahead are written

    for (int64_t g = g0, it = 0; g < g1; ++g, ++it) {
      walk.advance_to(g);
      BlockInfo bi;
      bi.seg_first = (g == g0) || (g == walk.bstart);
      bi.seg_last = (g == g1 - 1) || (g + 1 == walk.bend);
      bool ok = true;
      if (!TSC && bi.seg_first) {
        // rank-space query of this request into the permuted layout
        // qs[((h*2 + hi)*NCH + c)*4 + e] = q~[h][8c + 4hi + e]: four consecutive ranks
        // stay together, so it moves as float4, every load issued before the first store
        const float4* src = reinterpret_cast<const float4*>(p.qt) +
                            static_cast<size_t>(walk.b) * (S::H * S::RK / 4);
        constexpr int N4 = S::H * S::RK / 4, PER4 = (N4 + CT - 1) / CT;
        float4 q4[PER4];
#pragma unroll
        for (int u = 0; u < PER4; ++u)
          if (ctid + u * CT < N4) q4[u] = __ldcg(src + ctid + u * CT);
#pragma unroll
        for (int u = 0; u < PER4; ++u) {
          const int i4 = ctid + u * CT;
          if (i4 < N4) {
            const int h = (i4 * 4) / S::RK, k = (i4 * 4) % S::RK;
            const int c = k >> 3, hi = (k >> 2) & 1;
            *reinterpret_cast<float4*>(qs + ((h * 2 + hi) * NCH + c) * 4) = q4[u];
          }
        }
        named_bar_sync(1, CT);
      }
      const int ks = static_cast<int>(it % KST);
      float s[ROUNDS];
      int kph = 0;
      if constexpr (TSC) {
        // scores from the tensor cores: per round one 8-column load (this lane quarter's
        // head pair: term-major, head parity minor)
        const int sb = static_cast<int>(it & 1);
        ok = mbar_wait(&sfull[sb], (it >> 1) & 1, abort_flag, p.dev_err);
        ok = __all_sync(0xffffffffu, ok);   // TMEM loads are warp-collective
        bi.nvalid = ok ? sinfo[sb] : 0;
        if constexpr (SKIP) kph = sphys[sb];
        if (bi.seg_first) {
          ++nseg_c;
          const int qb = static_cast<int>((nseg_c - 1) & 1);
#pragma unroll
          for (int r = 0; r < ROUNDS; ++r) qf[r] = qinv[qb * S::H + head_of(r)];
          __syncwarp();
          if (lane == 0) mbar_arrive(&qfree[qb]);
        }
        tc_fence_after();
        float v[ROUNDS][8];
        if (ok) {
#pragma unroll
          for (int r = 0; r < ROUNDS; ++r)
            tmem_ld8(tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + L::SCOL +
                         sb * (S::H / 8) * 32 + ((cw / 4) * ROUNDS + r) * 32 + quarter * 8,
                     v[r]);
          tmem_wait_ld();
        }
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
          const float a = hl ? v[r][1] : v[r][0], b = hl ? v[r][3] : v[r][2];
          const float c = hl ? v[r][5] : v[r][4], d = hl ? v[r][7] : v[r][6];
          s[r] = ok ? ((a + b) + (c + d)) * qf[r] : -INFINITY;
          if constexpr (I4T)   // the key row's scale
            s[r] *= ksc[sb * S::H * kBlockSize + head_of(r) * kBlockSize + t];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[sb]);
      } else {
      ok = mbar_wait(&kfull[ks], (it / KST) & 1, abort_flag, p.dev_err);
      bi.nvalid = kinfo[ks];
      if constexpr (SKIP) kph = kphys[ks];
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        s[r] = -INFINITY;
        if (ok && head_ok(r)) {
          const int h = head_of(r);
          const uint8_t* kstage = kst + ks * L::KPS;   // this page's key stage
          // two packed fp32x2 accumulators = four independent chains
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          float kscale = 1.f;   // 4-bit pages: the key row's scale, applied to the dot product
          if constexpr (FMT == RCP_PAGES_INT4) {
            // r_k/2 bytes per key row: 8-byte chunks of 16 codes, rotated over the 16 lanes
            // so their rows' chunks spread over the banks; each 32-bit word holds codes
            // 8c .. 8c+7 (code 8c+i in nibble i).  A nibble n becomes the fp32 2^23 + (n ^ 8)
            // (exponent bits 0x4B000000), minus 2^23 + 8 the signed code, exactly.
            constexpr int RB = S::RK / 2, NU = RB / 8;
            const uint8_t* krow = kstage + (h * kBlockSize + t) * RB;
            kscale = __half2float(
                reinterpret_cast<const __half*>(kstage + Int4Page<S>::KCODES)[h * kBlockSize + t]);
            const float2 bias = make_float2(-8388616.f, -8388616.f);
#pragma unroll
            for (int v = 0; v < NU; ++v) {
              const int u = (v + t) % NU;
              const uint2 kv = *reinterpret_cast<const uint2*>(krow + u * 8);
              const uint32_t w2[2] = {kv.x, kv.y};
#pragma unroll
              for (int hw = 0; hw < 2; ++hw) {
                const int c = 2 * u + hw;
                const float4 qa = qs4[(h * 2 + 0) * NCH + c];
                const float4 qb = qs4[(h * 2 + 1) * NCH + c];
                const uint32_t w = w2[hw];
                float f[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  f[i] = __uint_as_float(((w >> (4 * i)) & 0xFu) ^ 0x4B000008u);
                acc0 = fma_f32x2(add_f32x2(make_float2(f[0], f[1]), bias), make_float2(qa.x, qa.y), acc0);
                acc1 = fma_f32x2(add_f32x2(make_float2(f[2], f[3]), bias), make_float2(qa.z, qa.w), acc1);
                acc0 = fma_f32x2(add_f32x2(make_float2(f[4], f[5]), bias), make_float2(qb.x, qb.y), acc0);
                acc1 = fma_f32x2(add_f32x2(make_float2(f[6], f[7]), bias), make_float2(qb.z, qb.w), acc1);
              }
            }
          } else if constexpr (F8) {
            // 16 E4M3 codes per 16-byte chunk; lanes 2u and 2u+1 start at chunk u so the
            // 16 tokens' 64-byte rows spread over all banks
            constexpr int NCH8 = S::RK / 16;
            const uint8_t* krow = kstage + (h * kBlockSize + t) * S::RK;
#pragma unroll
            for (int v = 0; v < NCH8; ++v) {
              const int c8 = (v + (t >> 1)) % NCH8;
              const uint4 kv = *reinterpret_cast<const uint4*>(krow + c8 * 16);
              const float4 qa0 = qs4[(h * 2 + 0) * NCH + 2 * c8];
              const float4 qb0 = qs4[(h * 2 + 1) * NCH + 2 * c8];
              const float4 qa1 = qs4[(h * 2 + 0) * NCH + 2 * c8 + 1];
              const float4 qb1 = qs4[(h * 2 + 1) * NCH + 2 * c8 + 1];
              const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
              const float4 qv[4] = {qa0, qb0, qa1, qb1};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float2 lo = e4m3x2_to_float2(static_cast<uint16_t>(w4[u] & 0xFFFFu));
                const float2 hi = e4m3x2_to_float2(static_cast<uint16_t>(w4[u] >> 16));
                acc0 = fma_f32x2(lo, make_float2(qv[u].x, qv[u].y), acc0);
                acc1 = fma_f32x2(hi, make_float2(qv[u].z, qv[u].w), acc1);
              }
            }
          } else {
            const __half* krow = reinterpret_cast<const __half*>(kstage) +
                                 (h * kBlockSize + t) * S::RK;
#pragma unroll
            for (int v = 0; v < NCH; ++v) {
              // swizzled stage: the same chunk for all lanes (q~ read as a broadcast);
              // otherwise a rotation keeps the 16 lanes on distinct banks
              const int c = KSWZ ? v : (v + t) % NCH;
              const uint4 kv = *reinterpret_cast<const uint4*>(
                  krow + (KSWZ ? ((c ^ (t & 7)) * 8) : c * 8));
              const float4 qa = qs4[(h * 2 + 0) * NCH + c];
              const float4 qb = qs4[(h * 2 + 1) * NCH + c];
              const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kv.x));
              const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kv.y));
              const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kv.z));
              const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kv.w));
              acc0 = fma_f32x2(k01, make_float2(qa.x, qa.y), acc0);
              acc1 = fma_f32x2(k23, make_float2(qa.z, qa.w), acc1);
              acc0 = fma_f32x2(k45, make_float2(qb.x, qb.y), acc0);
              acc1 = fma_f32x2(k67, make_float2(qb.z, qb.w), acc1);
            }
          }
          s[r] = (acc0.x + acc0.y) + (acc1.x + acc1.y);
          if constexpr (FMT == RCP_PAGES_INT4) s[r] *= kscale;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&kempty[ks]);
      }   // scores on the CUDA cores

      // online softmax (base 2), lazy rescale: the reference max only moves when a block
      // max exceeds it by more than kRescaleThreshold, so the accumulator is rarely touched
      // The ROUNDS independent butterflies advance level by level, so their shuffle
      // latencies overlap instead of adding up.
      __half ph[ROUNDS];
      float alpha[ROUNDS], sv[ROUNDS], bmax[ROUNDS], psum[ROUNDS], m_new[ROUNDS];
      bool valid[ROUNDS];
      bool need_any = false;
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        valid[r] = ok && head_ok(r) && t < bi.nvalid;
        sv[r] = valid[r] ? s[r] : -INFINITY;
        bmax[r] = sv[r];
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) {
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r)
          bmax[r] = fmaxf(bmax[r], __shfl_xor_sync(0xffffffffu, bmax[r], o));
      }
      // SKIP: the page is needed if one of this warp's heads has a score within skip_tau
      // of its running maximum (the first page of a segment always is)
      bool keep_mine = !SKIP;
      if constexpr (SKIP) {
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
          const float ref = bi.seg_first ? -INFINITY : mt[r];
          keep_mine |= head_ok(r) && !(bmax[r] < ref - p.skip_tau);
        }
      }
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        const float m_old = bi.seg_first ? -INFINITY : m_run[r];
        m_new[r] = (bmax[r] > m_old + kRescaleThreshold) ? bmax[r] : m_old;
        alpha[r] = (m_new[r] == m_old) ? 1.f : exp2f(m_old - m_new[r]);
        need_any |= (m_new[r] != m_old) && !bi.seg_first;
        const float pv = valid[r] ? exp2f(sv[r] - m_new[r]) : 0.f;
        ph[r] = __float2half_rn(pv);
        psum[r] = __half2float(ph[r]);
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) {
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) psum[r] += __shfl_xor_sync(0xffffffffu, psum[r], o);
      }
      // SKIP: the running state moves only once the page is known to be kept (computing
      // the weights before the vote measured faster than after it: it keeps the vote off
      // the path to the P write)
      float l_new[ROUNDS];
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        l_new[r] = (bi.seg_first ? 0.f : l_run[r] * alpha[r]) + psum[r];
        if constexpr (!SKIP) {
          l_run[r] = l_new[r];
          m_run[r] = m_new[r];
        }
      }
      const int fb = static_cast<int>(it & 1);
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        if (t == 0 && head_ok(r)) alpha_s[fb * HP + head_of(r)] = alpha[r];
      }
      const bool warp_need = __any_sync(0xffffffffu, need_any);
      const bool warp_keep = SKIP ? __any_sync(0xffffffffu, keep_mine) : true;
      if (lane == 0)
        flags_s[fb * NCW + cw] = (warp_need ? 1 : 0) | (*abort_flag ? 2 : 0) | (warp_keep ? 4 : 0);
      named_bar_sync(1, CT);
      int f = 0;
#pragma unroll
      for (int w2 = 0; w2 < NCW; ++w2) f |= flags_s[fb * NCW + w2];
      if (f & 2) {
        aborted = true;
        break;
      }
      const bool kept = !SKIP || (f & 4);
      if constexpr (SKIP) {
        if (ctid == 0 && p.page_kept != nullptr)
          p.page_kept[static_cast<int64_t>(walk.b) * p.bt_stride + (g - walk.bstart)] =
              kept ? 1 : 0;
        if (kept) {
          if (ctid == 0) {   // its value page: to the value-copy warp, as early as possible
            const int ds = static_cast<int>(nd % L::DS);
            if (nd < L::DS ||
                mbar_wait(&decempty[ds], ((nd / L::DS) - 1) & 1, abort_flag, p.dev_err)) {
              dec_s[ds] = kph;
              dec_n[ds] = bi.nvalid;
              mbar_arrive(&decfull[ds]);
            }
          }
          ++nd;
#pragma unroll
          for (int r = 0; r < ROUNDS; ++r) {
            l_run[r] = l_new[r];
            m_run[r] = m_new[r];
            mt[r] = bi.seg_first ? bmax[r] : fmaxf(mt[r], bmax[r]);
          }
        }
      }

      // P buffer / V stage order of this page among the accumulated ones
      const int64_t pi = SKIP ? kk : it;
      const int ps = static_cast<int>(pi % NPB);
      if (kept) {
      if (pi >= NPB) ok = mbar_wait(&pfree[ps], ((pi / NPB) - 1) & 1, abort_flag, p.dev_err) && ok;
      if (f & 1) {
        // rescale the accumulator columns after the previous block's MMAs have landed
        ok = mbar_wait(&pfree[(pi - 1) % NPB], ((pi - 1) / NPB) & 1, abort_flag, p.dev_err) && ok;
        ok = __all_sync(0xffffffffu, ok);   // TMEM loads / stores are warp-collective
        tc_fence_after();
        if (ok) {
#pragma unroll 1
          for (int i = chunk0; i < S::NCHUNK; i += CSTEP) {
#pragma unroll
            for (int hh = 0; hh < HP / 16; ++hh) {
              const uint32_t ta = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                  i * HP + hh * 16;
              float v[16];
              tmem_ld16(ta, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int h = hh * 16 + e;
                v[e] *= (h < S::H) ? alpha_s[fb * HP + h] : 1.f;
              }
              tmem_st16(ta, v);
            }
          }
          tmem_wait_st();
        }
      }
      // weights P (K-major, no swizzle): byte(h, t) = (h/8)*256 + (t/8)*128 + (h%8)*16 + (t%8)*2
      {
        uint8_t* pb = pbuf + ps * L::P_BYTES;
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
          if (head_ok(r)) {
            const int h = head_of(r);
            *reinterpret_cast<__half*>(pb + (h >> 3) * 256 + (t >> 3) * 128 + (h & 7) * 16 +
                                       (t & 7) * 2) = ph[r];
          }
        }
      }
      if (F8 && WB < S::NBOX) {
        // this block's remaining V boxes; the fp16 stage is free (pfree above covers the
        // MMA that read it two blocks ago)
        const int vr = static_cast<int>(it % VRS);
        ok = mbar_wait(&vfull[vr], (it / VRS) & 1, abort_flag, p.dev_err) && ok;
        widen_v_boxes<S, FMT, CT>(vraw + vr * L::VPS, vst + static_cast<int>(it % VST) * S::VSTAGE_BYTES,
                             bi.nvalid, WB, S::NBOX, ctid);
        __syncwarp();
        if (lane == 0) mbar_arrive(&vempty[vr]);
      }
      if (!F8 && bi.nvalid < kBlockSize) {
        // tokens past the sequence end (or a rejected block): zero their V rows so that
        // whatever those slots hold cannot reach the accumulator through 0 * NaN
        const int vs = static_cast<int>(pi % VST);
        ok = mbar_wait(&vfull[vs], (pi / VST) & 1, abort_flag, p.dev_err) && ok;
        const int nrow = kBlockSize - bi.nvalid;
        uint8_t* vb = vst + vs * S::VSTAGE_BYTES;
        for (int idx = ctid; idx < nrow * S::NBOX * 8; idx += CT) {
          const int row = bi.nvalid + idx / (S::NBOX * 8);
          const int rem = idx % (S::NBOX * 8);
          *reinterpret_cast<uint4*>(vb + (rem >> 3) * 2048 + row * 128 + (rem & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      if constexpr (SKIP)
        if (ctid == 0) pinfo[ps] = bi.seg_first ? 1 : 0;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[ps]);
      ++kk;
      }   // kept

      if (bi.seg_last) {
        // the segment's last accumulated page (a segment's first page is always kept)
        const int64_t last = SKIP ? kk - 1 : it;
        ok = mbar_wait(&pfree[last % NPB], (last / NPB) & 1, abort_flag, p.dev_err) && ok;
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        if (ok) {
          float* rec = p.rec + static_cast<size_t>(walk.b + cta) * S::REC;
#pragma unroll 1
          for (int i = chunk0; i < S::NCHUNK; i += CSTEP) {
            const int rrow = i * 128 + quarter * 32 + lane;
#pragma unroll
            for (int hh = 0; hh < HP / 16; ++hh) {
              const uint32_t ta = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                  i * HP + hh * 16;
              float v[16];
              tmem_ld16(ta, v);
              tmem_wait_ld();
              // head-major: the lanes of a warp (consecutive ranks) store 128 contiguous
              // bytes per head
              if (rrow < S::R) {
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  rec[static_cast<size_t>(hh * 16 + e) * S::R + rrow] = v[e];
              }
            }
          }
#pragma unroll
          for (int r = 0; r < ROUNDS; ++r) {
            if (t == 0 && head_ok(r)) {
              const int h = head_of(r);
              rec[static_cast<size_t>(S::R) * HP + h] = m_run[r];
              rec[static_cast<size_t>(S::R) * HP + HP + h] = l_run[r];
            }
          }
        }
        tc_fence_before();
      }
    }
    if constexpr (SKIP) {
      if (!aborted) {
        // no page follows: tell the MMA thread (the next P buffer's info word; its
        // previous use was read before the MMAs the last record waited for) and the
        // value-copy warp
        const int ps = static_cast<int>(kk % NPB);
        if (ctid == 0) {
          pinfo[ps] = -1;
          const int ds = static_cast<int>(nd % L::DS);
          if (nd < L::DS ||
              mbar_wait(&decempty[ds], ((nd / L::DS) - 1) & 1, abort_flag, p.dev_err)) {
            dec_s[ds] = -1;
            mbar_arrive(&decfull[ds]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[ps]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ----------------------------------------------------------------------------- launches
template <class S>
cudaError_t prepare_attn(int device) {
  (void)device;
  auto set = [](auto kernel, int smem) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  };
  cudaError_t e = set(decode_main_kernel<S, RCP_PAGES_FP16, false>, DecodeSmem<S, RCP_PAGES_FP16>::ALLOC);
  if (e == cudaSuccess)
    e = set(decode_main_kernel<S, RCP_PAGES_FP8_E4M3, false>,
            DecodeSmem<S, RCP_PAGES_FP8_E4M3>::ALLOC);
  if (e == cudaSuccess)
    e = set(decode_main_kernel<S, RCP_PAGES_INT4, false>, DecodeSmem<S, RCP_PAGES_INT4>::ALLOC);
  if (e == cudaSuccess)
    e = set(decode_main_kernel<S, RCP_PAGES_FP16, true>,
            DecodeSmem<S, RCP_PAGES_FP16, true>::ALLOC);
  if (e == cudaSuccess)
    e = set(decode_main_kernel<S, RCP_PAGES_FP8_E4M3, true>,
            DecodeSmem<S, RCP_PAGES_FP8_E4M3, true>::ALLOC);
  if (e == cudaSuccess)
    e = set(decode_main_kernel<S, RCP_PAGES_INT4, true>, DecodeSmem<S, RCP_PAGES_INT4, true>::ALLOC);
  return e;
}

// Launched as a programmatic dependent of the kernel before it (the query projection, with
// a decode step's append): its prologue and plan, and its page copies unless they read
// what an append in that launch writes, overlap that kernel.  With profiling events the
// plain stream order is kept so the events bracket decode_main exactly.
template <class S>
cudaError_t launch_attn(const CUtensorMap& tmap_v, const CUtensorMap& tmap_k, const AttnParams& p,
                        cudaStream_t stream, cudaEvent_t prof_start, cudaEvent_t prof_stop) {
  const bool pdl = prof_start == nullptr;
  cudaError_t e = cudaSuccess;
  if (prof_start && (e = cudaEventRecord(prof_start, stream)) != cudaSuccess) return e;
  constexpr int F16 = RCP_PAGES_FP16, E4M3 = RCP_PAGES_FP8_E4M3, I4 = RCP_PAGES_INT4;
  auto go = [&](auto kernel, int threads, int smem) {
    return launch_pdl(kernel, dim3(p.parts), dim3(threads), smem, stream, pdl, tmap_v, tmap_k, p);
  };
  if (p.page_format == E4M3)
    e = p.sparse ? go(decode_main_kernel<S, E4M3, true>, decode_threads<S, E4M3, true>(),
                      DecodeSmem<S, E4M3, true>::ALLOC)
                 : go(decode_main_kernel<S, E4M3, false>, decode_threads<S, E4M3>(),
                      DecodeSmem<S, E4M3>::ALLOC);
  else if (p.page_format == I4)
    e = p.sparse ? go(decode_main_kernel<S, I4, true>, decode_threads<S, I4, true>(),
                      DecodeSmem<S, I4, true>::ALLOC)
                 : go(decode_main_kernel<S, I4, false>, decode_threads<S, I4>(),
                      DecodeSmem<S, I4>::ALLOC);
  else
    e = p.sparse ? go(decode_main_kernel<S, F16, true>, decode_threads<S, F16, true>(),
                      DecodeSmem<S, F16, true>::ALLOC)
                 : go(decode_main_kernel<S, F16, false>, decode_threads<S, F16>(),
                      DecodeSmem<S, F16>::ALLOC);
  if (e != cudaSuccess) return e;
  if (prof_stop && (e = cudaEventRecord(prof_stop, stream)) != cudaSuccess) return e;
  return cudaSuccess;
}

// The chunked prefill's plan (one CTA).
template <class S>
cudaError_t launch_plan(const AttnParams& p, cudaStream_t stream, bool pdl) {
  return launch_pdl(plan_kernel<S>, dim3(1), dim3(kPlanThreads), 0, stream, pdl, p);
}

template cudaError_t launch_plan<ShapeMain>(const AttnParams&, cudaStream_t, bool);
template cudaError_t launch_plan<ShapeTiny>(const AttnParams&, cudaStream_t, bool);
template cudaError_t prepare_attn<ShapeMain>(int);
template cudaError_t prepare_attn<ShapeTiny>(int);
template cudaError_t launch_attn<ShapeMain>(const CUtensorMap&, const CUtensorMap&,
                                            const AttnParams&, cudaStream_t, cudaEvent_t,
                                            cudaEvent_t);
template cudaError_t launch_attn<ShapeTiny>(const CUtensorMap&, const CUtensorMap&,
                                            const AttnParams&, cudaStream_t, cudaEvent_t,
                                            cudaEvent_t);

}  // namespace rcp
