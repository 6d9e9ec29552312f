// Compile-time shapes, kernel parameter blocks and the workspace layout shared by the
// host launch code and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>

namespace rcp {

constexpr int kBlockSize = 16;   // tokens per page
constexpr int kMaxParts = 152;   // decode work partitions (CTAs) at most: one per SM of a
                                 // GB300; bounds the records the combine stages per tile

// Fewest blocks a decode work partition takes for a batch of nq requests (the split-K kernel
// and the merge derive the partition count from it alike).  With large pages (96 KiB of
// coefficients at (32, 128, 64, 1024)) a partition's 128 KiB split-K record must pay for
// itself: measured at batch 1 x 8192 tokens 45.2 / 43.8 / 48.0 us per step for 1 / 4 / 8
// blocks, at 16 x 1024 58.7 / 58.7 / 55.0 us.  Small pages spread over every partition.
template <class S>
__host__ __device__ constexpr int decode_min_pages(int nq) {
  return S::R >= 512 ? (nq >= 8 ? 8 : 4) : 1;
}

constexpr int pow2_at_least(int x, int lo) {
  int p = lo;
  while (p < x) p *= 2;
  return p;
}

// (H, d, r_k, R): heads, head dim, key rank per head, joint value rank.
template <int H_, int D_, int RK_, int R_>
struct Shape {
  static constexpr int H = H_, D = D_, RK = RK_, R = R_, BS = kBlockSize;
  static_assert(H % 4 == 0 && H <= 32, "heads are split over 4 compute warps, <= 32");
  static_assert(RK % 8 == 0 && R % 64 == 0 && D % 32 == 0 && D <= 256, "shape");
  static constexpr int HP = H <= 16 ? 16 : 32;          // heads padded to the MMA N
  static constexpr int NCHUNK = (R + 127) / 128;        // M = 128 chunks of the value rank
  static constexpr int NBOX = R / 64;                   // 64-wide tensor boxes per V page
  static constexpr int TMEM_COLS = pow2_at_least(NCHUNK * HP, 32);
  static constexpr int KPAGE_BYTES = H * BS * RK * 2;   // one block of K coefficients
  static constexpr int VPAGE_BYTES = BS * R * 2;        // one block of V coefficients
  static constexpr int VSTAGE_BYTES = NCHUNK * 2 * 2048;  // smem A operand of NCHUNK MMAs
  // floats in one split-K partial record: the accumulator head-major [HP][R], then the
  // running maximum m[HP] and sum l[HP]
  static constexpr int REC = R * HP + 2 * HP;
  static_assert(NCHUNK * HP <= 512, "accumulator must fit in tensor memory");
};

// 4-bit pages: bytes of one K page (codes [H][16][r_k/2], then fp16 scales [H][16]) and of
// one V page (codes [16][R/2], then fp16 scales [16][R/64]).
template <class S>
struct Int4Page {
  static constexpr int64_t KCODES = S::H * kBlockSize * S::RK / 2;
  static constexpr int64_t KBYTES = KCODES + S::H * kBlockSize * 2;
  static constexpr int64_t VCODES = kBlockSize * S::R / 2;
  static constexpr int64_t VBYTES = VCODES + kBlockSize * (S::R / 64) * 2;
};

using ShapeMain = Shape<32, 128, 64, 1024>;
using ShapeTiny = Shape<4, 64, 16, 64>;

// Split-K combine + W_v up-projection (combine.cu): tiles of NT requests; the value rank R
// is cut into KSPLIT slices of KB 64-wide k-blocks (RANKS ranks), one CTA per (tile, head,
// slice).  The records a tile's requests own (at most REC_ROWS: NT requests over at most
// kMaxParts partitions) stream through NBUF tensor copies of CHUNK records.
template <class S>
struct CombineCfg {
  static constexpr int NT = 64;
  static constexpr int KSPLIT = (S::R / 64) < 8 ? (S::R / 64) : 8;
  static constexpr int KB = (S::R / 64) / KSPLIT;
  static constexpr int RANKS = KB * 64;
  static constexpr int REC_ROWS = NT + kMaxParts;
  static constexpr int CHUNK = 32, NBUF = 2;
  static_assert((S::R / 64) % KSPLIT == 0, "combine slices");
};

// Chunked prefill: 128 query rows x 128 keys per tile; the value rank is cut into slices
// of at most 256 (one CTA each, clustered); key rank padded to 64 (one 128-byte row).
template <class S>
struct PrefillCfg {
  static constexpr int QT = 128, KT = 128;
  static constexpr int RQ = S::R >= 256 ? 256 : S::R;
  static constexpr int NQ = S::R / RQ;
  static constexpr int RKP = 64;
  static_assert(S::R % RQ == 0 && RQ % 64 == 0 && S::RK <= 64 && S::D % 64 == 0, "prefill shape");
};

// Reconstructing prefill: V^ = C_v W_v for every cached key of the batch, 256 keys (16
// pages) x 256 columns of H*d per CTA pair (a 2-CTA cluster: 128 keys and 128 of the W_v
// columns staged in each CTA), K = R in 64-wide k-blocks, STG pipeline stages.
template <class S>
struct ReconCfg {
  static constexpr int MT = 128, NT = 256, NTC = NT / 2, KB = S::R / 64, STG = 6;
  static_assert((S::H * S::D) % NT == 0 && S::R % 64 == 0, "reconstruct tiling");
};

// Upper bound on 128-row prefill query tiles for nq query rows (each request with rows
// adds at most one partial tile, and at most nq requests have rows).
inline int64_t prefill_max_tiles(int64_t nq) { return (nq + 127) / 128 + nq; }

// Workspace carve-up for nq query rows (all offsets 256-byte aligned).
struct WsLayout {
  size_t cum, qlen, qrow, qt, rec, upart, ucnt, tile_b, tile_qt, tcount, total;
};
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
template <class S>
inline WsLayout ws_layout(int64_t nq) {
  WsLayout w{};
  size_t o = 0;
  w.cum = o;  o = align256(o + sizeof(int64_t) * (nq + 1));
  w.qlen = o; o = align256(o + sizeof(int32_t) * nq);
  w.qrow = o; o = align256(o + sizeof(int32_t) * nq);
  // rank-space queries: fp32 [nq][H][r_k] (decode) or fp16 hi + lo [nq][H][64] (prefill)
  const size_t qt_row = static_cast<size_t>(S::H) * (S::RK > 64 ? S::RK : 64) * 4;
  w.qt = o;   o = align256(o + qt_row * nq);
  w.tile_b = o;  o = align256(o + sizeof(int32_t) * prefill_max_tiles(nq));
  w.tile_qt = o; o = align256(o + sizeof(int32_t) * prefill_max_tiles(nq));
  w.tcount = o;  o = align256(o + sizeof(int32_t));
  // decode only from here on: split-K partial records, one per (request, partition)
  // segment, at index request + partition
  w.rec = o;  o = align256(o + sizeof(float) * (nq + kMaxParts) * static_cast<size_t>(S::REC));
  // the combine's fp32 partial outputs [tile][head][slice][NT][128] and its counter per
  // (tile, head)
  const size_t tiles = static_cast<size_t>((nq + CombineCfg<S>::NT - 1) / CombineCfg<S>::NT);
  w.upart = o;
  o = align256(o + sizeof(float) * tiles * S::H * CombineCfg<S>::KSPLIT * CombineCfg<S>::NT * 128);
  w.ucnt = o; o = align256(o + sizeof(int32_t) * tiles * S::H);
  w.total = o;
  return w;
}

// The reconstructing prefill never uses the decode-only region at the end (rec):
// its per-request block prefix sums and the reconstructed values V^ start where they
// start, for at most batch x max_blocks_per_seq pages.
struct ReconLayout {
  size_t vcum, vhat, kw, vw, tw, total;
};
// widen (E4M3 pages): also fp16 copies of the pages the batch reads, [pages][H][16][r_k]
// and [pages][16][R], and the block table re-addressed to them, [batch][max_blocks].
template <class S>
inline ReconLayout recon_layout(int64_t nq, int64_t batch, int64_t max_blocks, bool widen = false) {
  const WsLayout w = ws_layout<S>(nq);
  const size_t pages = static_cast<size_t>(batch) * max_blocks;
  ReconLayout r;
  size_t o = w.rec;
  r.vcum = o;  o = align256(o + sizeof(int64_t) * (batch + 1));
  r.vhat = o;  o = align256(o + 2 * pages * kBlockSize * S::H * S::D);
  r.kw = r.vw = r.tw = 0;
  if (widen) {
    r.kw = o;  o = align256(o + 2 * pages * S::H * kBlockSize * S::RK);
    r.vw = o;  o = align256(o + 2 * pages * kBlockSize * S::R);
    r.tw = o;  o = align256(o + sizeof(int32_t) * pages);
  }
  r.total = o > w.total ? o : w.total;
  return r;
}

// Everything the attention kernels of one call see.
struct AttnParams {
  const void* q;              // [nq][H][d] fp16
  const void* U_k;            // [H][r_k][d] fp16
  const void* W_v;            // [R][H*d] fp16
  const void* k_pages;        // [num_blocks][H][16][r_k] fp16 (or E4M3 codes)
  const void* v_pages;        // [num_blocks][16][R] fp16 (or E4M3 codes)
  const int32_t* block_table; // [rows][bt_stride]
  const int32_t* seq_lens;    // [batch]
  const int32_t* cu_chunk;    // prefill: [batch+1]; decode: nullptr
  void* out;                  // [nq][H][d] fp16
  uint32_t* dev_err;
  // workspace regions
  int64_t* cum;               // [nq+1] prefix sums of blocks per query row (decode: written
                              // by partition 0 of the split-K kernel for the combine)
  int32_t* qlen;              // [nq] keys attended by each query row (prefill plan)
  int32_t* qrow;              // [nq] block-table row of each query row (prefill plan)
  float* qt;                  // [nq][H][r_k] rank-space queries, scaled by log2(e)/sqrt(d)
  float* rec;                 // [(nq + parts)][REC] split partials
  int32_t* ucnt;              // decode: [tiles][H] combine counters, zeroed by partition 0
  // prefill only (nullptr for decode)
  int32_t* tile_b;            // [max tiles] request of each 128-row query tile
  int32_t* tile_qt;           // [max tiles] tile index within its request
  int32_t* tcount;            // [1] number of query tiles
  void* qhi;                  // [nq][H][64] fp16 rank-space queries (scaled), zero past r_k
  void* qlo;                  // [nq][H][64] fp16 remainder q~ - qhi
  // reconstructing prefill only (nullptr otherwise)
  int64_t* vcum;              // [batch+1] prefix sums of blocks per request
  void* vhat;                 // [sum of blocks * 16][H*d] fp16 reconstructed values C_v W_v
  int64_t num_blocks;
  int32_t bt_stride;          // max_blocks_per_seq
  int32_t batch;
  int32_t nq;
  int32_t parts;              // decode CTAs (work partitions)
  int32_t page_format;        // RCP_PAGES_* of the pages the kernels read
  // block-sparse decode: a page whose every head's largest score is more than skip_tau
  // (log2 units) below that head's running maximum is left out, values unread
  int32_t sparse;
  float skip_tau;
  uint8_t* page_kept;         // sparse, optional: [rows][bt_stride], 1 = page read, 0 = skipped
  // decode step: the slots the step's own append writes (the kernel before the split-K
  // kernel); a partition waits for the append before it copies a page among them
  const int64_t* slots;
  int32_t n_slots;
  float qscale;               // log2(e) / sqrt(d)
};

// What the split-K combine + up-projection of a decode call sees (combine.cu).
struct CombineParams {
  const int64_t* cum;         // [nq+1] block prefix sums, written by the split-K kernel
  const float* rec;           // [(nq + parts)][REC] partial records (head-major accumulator,
                              // then m[HP], l[HP]), record id = request + partition
  float* upart;               // [tiles][H][KSPLIT][NT][128] fp32 partial outputs
  int32_t* ucnt;              // [tiles][H] arrivals, zero on entry
  void* out;                  // [nq][H][d] fp16
  uint32_t* dev_err;
  int32_t nq;
  int32_t parts;              // split-K partitions launched
};

struct AppendParams {
  const void* k;              // [T][H][d] fp16
  const void* v;              // [T][H*d] fp16
  const int64_t* slots;       // [T]
  const void* U_k;
  const void* W_v;
  void* k_pages;
  void* v_pages;
  uint32_t* dev_err;
  int64_t num_blocks;
  int32_t T;
  int32_t page_format;        // RCP_PAGES_*: fp16, E4M3 or 4-bit codes with scales
  // the rank-space queries are projected in the same launch (nq = 0: none): decode as fp32
  // into qt, or (qhi != nullptr) a prefill chunk's as fp16 (hi, lo) pairs into qhi / qlo
  float* qt;                  // [nq][H][r_k] fp32, q~ scaled by qscale
  void* qhi;                  // [nq][H][64] fp16 each, zero past r_k
  void* qlo;
  int32_t nq;
  float qscale;
  // wait for the launch before this one only at exit (that launch writes nothing this
  // one reads or writes), so that both run at once
  int32_t wait_at_exit;
};

}  // namespace rcp
