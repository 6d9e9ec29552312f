// C ABI of the rank-compressed paged attention library: handle, host block pool,
// argument checks, tensor-map set-up and kernel dispatch by shape.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <climits>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "launch.h"
#include "rcp.h"
#include "shape.h"

using rcp::ShapeMain;
using rcp::ShapeTiny;

enum ShapeId { kShapeNone = -1, kShapeMain = 0, kShapeTiny = 1 };

struct rcp_cache {
  rcp_cache_config cfg;
  void* k_pages;
  void* v_pages;
  const void* U_k;
  const void* W_v;
  uint32_t* dev_err;
  int shape;
  std::vector<int32_t> free_ids;   // LIFO stack of free physical blocks
  std::vector<uint8_t> is_free;
  // device-side state, set up at the first kernel call on a device
  int device;
  int num_sms;
  CUtensorMap tmap_v;       // V pages as [num_blocks*16][R], 64 x 16 boxes (decode A operand)
  CUtensorMap tmap_wv_k;    // W_v as [R][H*d], 64 x 128 boxes (append: K-major A)
  CUtensorMap tmap_wv_mn;   // W_v as [R][H*d], 64 x 64 boxes (up-projection: MN-major A)
  CUtensorMap tmap_uk64;    // U_k as [H*r_k][d], 64 x 64 boxes (key and query pairs: A)
  CUtensorMap tmap_kp;      // K pages as [num_blocks*H*16][r_k], 64 x 16 boxes (prefill B)
  CUtensorMap tmap_kpage;   // the same rows, 64 x 256 boxes (decode: half a page per box;
                            // E4M3 pages: bytes, 64-byte swizzle)
  // optional events recorded around the split-K attention kernel
  cudaEvent_t prof_start;
  cudaEvent_t prof_stop;
};

namespace {

int shape_of(const rcp_cache_config* c) {
  if (c->block_size != rcp::kBlockSize) return kShapeNone;
  if (c->num_heads == ShapeMain::H && c->head_dim == ShapeMain::D && c->rank_k == ShapeMain::RK &&
      c->rank_v == ShapeMain::R)
    return kShapeMain;
  if (c->num_heads == ShapeTiny::H && c->head_dim == ShapeTiny::D && c->rank_k == ShapeTiny::RK &&
      c->rank_v == ShapeTiny::R)
    return kShapeTiny;
  return kShapeNone;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  fn = reinterpret_cast<EncodeTiledFn>(ptr);
  return fn;
}

// A 2-D fp16 tensor map with 128-byte swizzle: `inner` elements per row (contiguous),
// `rows` rows `row_bytes` apart, boxes of box_inner x box_rows.
bool encode_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 2-D byte tensor map with 64-byte swizzle (E4M3 key pages with 64-byte rows: the
// decode's tensor-core scoring reads them as the swizzled K-major operand).
bool encode_2d_u8_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(inner), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 2-D fp32 tensor map without swizzle (the split-K records for the combine).
bool encode_2d_f32(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The combine's tensor maps over the records of nq query rows: slices of one head's ranks
// of a CTA, and 4-float groups of (m, l).
template <class S>
bool encode_records(CUtensorMap* slices, CUtensorMap* ml, const float* rec, int64_t nq) {
  using U = rcp::CombineCfg<S>;
  const uint64_t rows = static_cast<uint64_t>(nq) + rcp::kMaxParts;
  const uint64_t inner = S::REC, bytes = static_cast<uint64_t>(S::REC) * 4;
  return encode_2d_f32(slices, rec, inner, rows, bytes, U::RANKS, U::CHUNK) &&
         encode_2d_f32(ml, rec, inner, rows, bytes, 4, U::REC_ROWS);
}

template <class S>
cudaError_t prepare_kernels(int dev) {
  cudaError_t e = rcp::prepare_attn<S>(dev);
  if (e == cudaSuccess) e = rcp::prepare_gemm<S>();
  if (e == cudaSuccess) e = rcp::prepare_combine<S>();
  if (e == cudaSuccess) e = rcp::prepare_prefill<S>();
  if (e == cudaSuccess) e = rcp::prepare_recon<S>();
  return e;
}

// Device set-up on first use per device: SM count, kernel attributes and the tensor maps
// of the buffers the handle owns pointers to (V pages, W_v twice, U_k).
rcp_status ensure_device(rcp_cache* c) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return RCP_ERR_CUDA;
  if (dev == c->device) return RCP_OK;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return RCP_ERR_CUDA;
  cudaError_t e = c->shape == kShapeMain ? prepare_kernels<ShapeMain>(dev)
                                         : prepare_kernels<ShapeTiny>(dev);
  if (e != cudaSuccess) return RCP_ERR_CUDA;
  const rcp_cache_config& g = c->cfg;
  const uint64_t hd = static_cast<uint64_t>(g.num_heads) * g.head_dim;
  if (!encode_2d(&c->tmap_v, c->v_pages, g.rank_v, static_cast<uint64_t>(g.num_blocks) * 16,
                 static_cast<uint64_t>(g.rank_v) * 2, 64, 16) ||
      !encode_2d(&c->tmap_wv_k, c->W_v, hd, g.rank_v, hd * 2, 64, 128) ||
      !encode_2d(&c->tmap_wv_mn, c->W_v, hd, g.rank_v, hd * 2, 64, 64) ||
      !encode_2d(&c->tmap_uk64, c->U_k, g.head_dim,
                 static_cast<uint64_t>(g.num_heads) * g.rank_k, static_cast<uint64_t>(g.head_dim) * 2,
                 64, 64) ||
      !encode_2d(&c->tmap_kp, c->k_pages, g.rank_k,
                 static_cast<uint64_t>(g.num_blocks) * g.num_heads * 16,
                 static_cast<uint64_t>(g.rank_k) * 2, 64, 16) ||
      !encode_2d(&c->tmap_kpage, c->k_pages, g.rank_k,
                 static_cast<uint64_t>(g.num_blocks) * g.num_heads * 16,
                 static_cast<uint64_t>(g.rank_k) * 2, 64,
                 g.num_heads * 16 < 256 ? static_cast<uint32_t>(g.num_heads * 16) : 256))
    return RCP_ERR_CUDA;
  // E4M3 key pages with 64-byte rows: the decode copies them through a byte map
  if (g.page_format == RCP_PAGES_FP8_E4M3 && g.rank_k == 64 &&
      !encode_2d_u8_sw64(&c->tmap_kpage, c->k_pages, 64,
                         static_cast<uint64_t>(g.num_blocks) * g.num_heads * 16,
                         g.num_heads * 16 < 256 ? static_cast<uint32_t>(g.num_heads * 16) : 256))
    return RCP_ERR_CUDA;
  c->num_sms = sms;
  c->device = dev;
  return RCP_OK;
}

template <class S>
size_t ws_bytes_for(int64_t nq) {
  return rcp::ws_layout<S>(nq).total;
}

size_t ws_bytes(const rcp_cache* c, int64_t nq) {
  return c->shape == kShapeMain ? ws_bytes_for<ShapeMain>(nq) : ws_bytes_for<ShapeTiny>(nq);
}

template <class S>
void fill_ws(rcp::AttnParams& p, void* ws, int64_t nq) {
  using S_ = S;
  const rcp::WsLayout w = rcp::ws_layout<S>(nq);
  uint8_t* b = static_cast<uint8_t*>(ws);
  p.cum = reinterpret_cast<int64_t*>(b + w.cum);
  p.qlen = reinterpret_cast<int32_t*>(b + w.qlen);
  p.qrow = reinterpret_cast<int32_t*>(b + w.qrow);
  p.qt = reinterpret_cast<float*>(b + w.qt);
  p.rec = reinterpret_cast<float*>(b + w.rec);
  p.ucnt = reinterpret_cast<int32_t*>(b + w.ucnt);
  p.tile_b = reinterpret_cast<int32_t*>(b + w.tile_b);
  p.tile_qt = reinterpret_cast<int32_t*>(b + w.tile_qt);
  p.tcount = reinterpret_cast<int32_t*>(b + w.tcount);
  // prefill queries reuse the decode query region: hi then lo, [nq][H][64] fp16 each
  p.qhi = b + w.qt;
  p.qlo = b + w.qt + static_cast<size_t>(nq) * S::H * 64 * 2;
  p.vcum = nullptr;
  p.vhat = nullptr;
}

// E4M3 pages: fp16 copies of the batch's pages for the reconstructing prefill
struct Widened {
  void* k16;
  void* v16;
  int32_t* table16;
};

template <class S>
Widened fill_recon(rcp::AttnParams& p, void* ws, int64_t nq, int64_t batch, int64_t max_blocks,
                   bool widen) {
  const rcp::ReconLayout r = rcp::recon_layout<S>(nq, batch, max_blocks, widen);
  uint8_t* b = static_cast<uint8_t*>(ws);
  p.vcum = reinterpret_cast<int64_t*>(b + r.vcum);
  p.vhat = b + r.vhat;
  if (!widen) return Widened{nullptr, nullptr, nullptr};
  return Widened{b + r.kw, b + r.vw, reinterpret_cast<int32_t*>(b + r.tw)};
}

size_t recon_ws_bytes(const rcp_cache* c, int64_t nq, int64_t batch, int64_t max_blocks) {
  const bool widen = c->cfg.page_format != RCP_PAGES_FP16;
  return c->shape == kShapeMain ? rcp::recon_layout<ShapeMain>(nq, batch, max_blocks, widen).total
                                : rcp::recon_layout<ShapeTiny>(nq, batch, max_blocks, widen).total;
}

// Block-sparse decode options (rcp_decode_attn_sparse).
struct SparseArgs {
  float tau;            // log2 units, +inf leaves no page out
  uint8_t* page_kept;
};

// New tokens a decode step appends before its attention (rcp_decode_step).
struct AppendArgs {
  const void* k;
  const void* v;
  const int64_t* slots;
  int32_t T;
};

rcp_status check_append(const AppendArgs& a) {
  if (a.T < 0) return RCP_ERR_INVALID_ARG;
  if (a.T == 0) return RCP_OK;
  if (!a.k || !a.v || !a.slots) return RCP_ERR_INVALID_ARG;
  if (!aligned16(a.k) || !aligned16(a.v) || (reinterpret_cast<uintptr_t>(a.slots) & 7u))
    return RCP_ERR_INVALID_ARG;
  return RCP_OK;
}

// The projection launch: a step's append (app->T tokens; none when app is null) and, when
// nq > 0, the rank-space queries q~: a decode's (fp32 into qt) or, when qhi is set, a
// chunked prefill's (fp16 hi / lo pairs), as tcgen05 jobs of one grid.  wait_at_exit: the
// launch before this one writes nothing this one touches, and is waited for only at exit.
rcp_status launch_front(rcp_cache* c, const AppendArgs* app, const void* q, int32_t nq,
                        float* qt, float qscale, cudaStream_t s, void* qhi = nullptr,
                        void* qlo = nullptr, bool wait_at_exit = false) {
  const int32_t T = app ? app->T : 0;
  if (T == 0 && nq == 0) return RCP_OK;
  rcp::AppendParams p{};
  p.k = T ? app->k : nullptr;
  p.v = T ? app->v : nullptr;
  p.slots = T ? app->slots : nullptr;
  p.U_k = c->U_k;
  p.W_v = c->W_v;
  p.k_pages = c->k_pages;
  p.v_pages = c->v_pages;
  p.dev_err = c->dev_err;
  p.num_blocks = c->cfg.num_blocks;
  p.T = T;
  p.page_format = c->cfg.page_format;
  p.qt = qt;
  p.qhi = qhi;
  p.qlo = qlo;
  p.nq = nq;
  p.qscale = qscale;
  p.wait_at_exit = wait_at_exit ? 1 : 0;
  // the new tokens' k and v and the queries as [rows][H*d] B operands (16-row tiles up to
  // 16 rows, 64-row tiles up to 256, else 256-row tiles); an absent operand takes another's
  // map (never read)
  const uint64_t hd = static_cast<uint64_t>(c->cfg.num_heads) * c->cfg.head_dim;
  const int32_t rows = T > nq ? T : nq;
  const uint32_t nt = rows <= 16 ? 16 : (rows <= 256 ? 64 : 256);
  CUtensorMap vmap, kmap, qmap;
  if (T > 0 && (!encode_2d(&vmap, app->v, hd, static_cast<uint64_t>(T), hd * 2, 64, nt) ||
                !encode_2d(&kmap, app->k, hd, static_cast<uint64_t>(T), hd * 2, 64, nt)))
    return RCP_ERR_CUDA;
  if (nq > 0 && !encode_2d(&qmap, q, hd, static_cast<uint64_t>(nq), hd * 2, 64, nt))
    return RCP_ERR_CUDA;
  if (T == 0) vmap = kmap = qmap;
  if (nq == 0) qmap = kmap;
  const cudaError_t e =
      c->shape == kShapeMain
          ? rcp::launch_append_gemm<ShapeMain>(c->tmap_wv_k, c->tmap_uk64, vmap, kmap, qmap, p, s)
          : rcp::launch_append_gemm<ShapeTiny>(c->tmap_wv_k, c->tmap_uk64, vmap, kmap, qmap, p, s);
  return e == cudaSuccess ? RCP_OK : RCP_ERR_CUDA;
}

rcp_status run_attention(rcp_cache* c, const void* q, const int32_t* cu_chunk, int32_t nq,
                         const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, int32_t batch, void* out, void* ws,
                         size_t ws_size, rcp_stream stream, const AppendArgs* app = nullptr,
                         bool recon = false, const SparseArgs* sparse = nullptr) {
  if (!c || batch < 0 || nq < 0 || max_blocks_per_seq < 1) return RCP_ERR_INVALID_ARG;
  if (app && check_append(*app) != RCP_OK) return RCP_ERR_INVALID_ARG;
  if (nq == 0) {
    // nothing to attend; a step still appends its tokens
    if (!app || app->T == 0) return RCP_OK;
    rcp_status st = ensure_device(c);
    if (st != RCP_OK) return st;
    return launch_front(c, app, nullptr, 0, nullptr, 0.f, static_cast<cudaStream_t>(stream));
  }
  if (batch == 0 && cu_chunk) return RCP_ERR_INVALID_ARG;
  if (!q || !block_table || !seq_lens || !out || !ws) return RCP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (cu_chunk && (reinterpret_cast<uintptr_t>(cu_chunk) & 3u)))
    return RCP_ERR_INVALID_ARG;
  // a prefill on quantized pages widens the pages it reads into the workspace (both variants)
  const bool paged_ws = recon || (cu_chunk && c->cfg.page_format != RCP_PAGES_FP16);
  if (ws_size < (paged_ws ? recon_ws_bytes(c, nq, batch, max_blocks_per_seq) : ws_bytes(c, nq)))
    return RCP_ERR_WORKSPACE;
  // block-sparse skipping is a decode option
  if (sparse && cu_chunk) return RCP_ERR_UNSUPPORTED;
  rcp_status st = ensure_device(c);
  if (st != RCP_OK) return st;
  rcp::AttnParams p{};
  p.q = q;
  p.U_k = c->U_k;
  p.W_v = c->W_v;
  p.k_pages = c->k_pages;
  p.v_pages = c->v_pages;
  p.page_format = c->cfg.page_format;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.cu_chunk = cu_chunk;
  p.out = out;
  p.dev_err = c->dev_err;
  p.num_blocks = c->cfg.num_blocks;
  p.bt_stride = max_blocks_per_seq;
  p.batch = batch;
  p.nq = nq;
  // work partitions: one CTA per SM, never more than the blocks that can exist
  const int64_t max_blocks_total = static_cast<int64_t>(nq) * max_blocks_per_seq;
  int64_t parts = c->num_sms < rcp::kMaxParts ? c->num_sms : rcp::kMaxParts;
  if (parts > max_blocks_total) parts = max_blocks_total;
  if (parts < 1) parts = 1;
  p.parts = static_cast<int32_t>(parts);
  p.slots = app && app->T > 0 ? app->slots : nullptr;
  p.n_slots = app ? app->T : 0;
  p.sparse = sparse ? 1 : 0;
  p.skip_tau = sparse ? sparse->tau : 0.f;
  p.page_kept = sparse ? sparse->page_kept : nullptr;
  p.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(c->cfg.head_dim)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (c->shape == kShapeMain) fill_ws<ShapeMain>(p, ws, nq);
  else fill_ws<ShapeTiny>(p, ws, nq);
  const bool pdl = c->prof_start == nullptr;
  // the prefill kernels read fp16 pages; E4M3 and 4-bit pages are widened first into the
  // workspace, which is then sized by the pages the batch can reach
  if (cu_chunk) {
    // chunked prefill: plan + fp16 rank-space queries, then the tiled tensor-core kernel
    const uint64_t hq = static_cast<uint64_t>(c->cfg.num_heads) * 64;
    CUtensorMap qhi_map, qlo_map;
    if (static_cast<int64_t>(c->cfg.num_blocks) * c->cfg.num_heads * 16 >= (int64_t{1} << 31))
      return RCP_ERR_UNSUPPORTED;
    if (!encode_2d(&qhi_map, p.qhi, hq, static_cast<uint64_t>(nq), hq * 2, 64, 128) ||
        !encode_2d(&qlo_map, p.qlo, hq, static_cast<uint64_t>(nq), hq * 2, 64, 128))
      return RCP_ERR_CUDA;
    const int max_tiles = static_cast<int>((nq + 127) / 128 + (batch < nq ? batch : nq));
    const uint64_t hdq = static_cast<uint64_t>(c->cfg.num_heads) * c->cfg.head_dim;
    CUtensorMap q_map;
    if (!encode_2d(&q_map, q, hdq, static_cast<uint64_t>(nq), hdq * 2, 64, nq <= 256 ? 64 : 256))
      return RCP_ERR_CUDA;
    // reconstructing variant: V^ rows for at most batch x max_blocks_per_seq pages
    const int64_t max_pages = static_cast<int64_t>(batch) * max_blocks_per_seq;
    const bool widen = p.page_format != RCP_PAGES_FP16;
    CUtensorMap vhat_map = c->tmap_v, kp16_map = c->tmap_kp, vp16_map = c->tmap_v;
    Widened wd{nullptr, nullptr, nullptr};
    rcp::AttnParams pw = p;   // the widening pass reads the cache's own pages and table
    if (recon || widen) {
      if (max_pages * 16 >= (int64_t{1} << 31)) return RCP_ERR_UNSUPPORTED;
      if (widen && max_pages * c->cfg.num_heads * 16 >= (int64_t{1} << 31)) return RCP_ERR_UNSUPPORTED;
      wd = c->shape == kShapeMain
               ? fill_recon<ShapeMain>(p, ws, nq, batch, max_blocks_per_seq, widen)
               : fill_recon<ShapeTiny>(p, ws, nq, batch, max_blocks_per_seq, widen);
      if (recon && !encode_2d(&vhat_map, p.vhat, hdq, static_cast<uint64_t>(max_pages) * 16,
                              hdq * 2, 64, 128))
        return RCP_ERR_CUDA;
      if (widen) {
        pw = p;   // with the plan's page prefix sums
        const uint64_t rk = c->cfg.rank_k, rv = c->cfg.rank_v;
        if (!encode_2d(&kp16_map, wd.k16, rk,
                       static_cast<uint64_t>(max_pages) * c->cfg.num_heads * 16, rk * 2, 64, 16) ||
            !encode_2d(&vp16_map, wd.v16, rv, static_cast<uint64_t>(max_pages) * 16, rv * 2, 64, 16))
          return RCP_ERR_CUDA;
        // the kernels after the widening pass read the fp16 copies
        p.k_pages = wd.k16;
        p.v_pages = wd.v16;
        p.block_table = wd.table16;
        p.num_blocks = max_pages;
        p.page_format = RCP_PAGES_FP16;
      }
    }
    const CUtensorMap& vals = recon ? vhat_map : widen ? vp16_map : c->tmap_v;
    const CUtensorMap& kmap = widen ? kp16_map : c->tmap_kp;
    const CUtensorMap& vsrc = widen ? vp16_map : c->tmap_v;
    // a step with the chunk's append: the plan first, then one projection launch for the
    // append and the chunk's queries, which runs beside the plan (it waits for the plan
    // only at exit: the plan writes the workspace's plan arrays, the projections the pages
    // and the query pairs)
    const bool fused = app && app->T > 0;
    if (c->shape == kShapeMain) {
      e = rcp::launch_plan<ShapeMain>(p, s, pdl);
      if (e == cudaSuccess && fused) {
        if (launch_front(c, app, q, nq, nullptr, p.qscale, s, p.qhi, p.qlo, pdl) != RCP_OK)
          return RCP_ERR_CUDA;
      } else if (e == cudaSuccess) {
        e = rcp::launch_qproj_gemm<ShapeMain>(c->tmap_uk64, q_map, p.qhi, p.qlo, nq, p.qscale,
                                              c->dev_err, s, pdl);
      }
      // profiling events bracket the attention proper: reconstruction + prefill kernel
      if (e == cudaSuccess && c->prof_start) e = cudaEventRecord(c->prof_start, s);
      if (e == cudaSuccess && widen)
        e = rcp::launch_widen<ShapeMain>(pw, wd.k16, wd.v16, wd.table16, max_pages, c->num_sms, s,
                                         pdl);
      if (e == cudaSuccess && recon)
        e = rcp::launch_recon<ShapeMain>(vsrc, c->tmap_wv_mn, p, max_pages, c->num_sms, s, pdl);
      if (e == cudaSuccess)
        e = rcp::launch_prefill<ShapeMain>(qhi_map, qlo_map, kmap, vals, c->tmap_wv_mn, p,
                                           max_tiles, s, pdl, recon);
    } else {
      e = rcp::launch_plan<ShapeTiny>(p, s, pdl);
      if (e == cudaSuccess && fused) {
        if (launch_front(c, app, q, nq, nullptr, p.qscale, s, p.qhi, p.qlo, pdl) != RCP_OK)
          return RCP_ERR_CUDA;
      } else if (e == cudaSuccess) {
        e = rcp::launch_qproj_gemm<ShapeTiny>(c->tmap_uk64, q_map, p.qhi, p.qlo, nq, p.qscale,
                                              c->dev_err, s, pdl);
      }
      // profiling events bracket the attention proper: reconstruction + prefill kernel
      if (e == cudaSuccess && c->prof_start) e = cudaEventRecord(c->prof_start, s);
      if (e == cudaSuccess && widen)
        e = rcp::launch_widen<ShapeTiny>(pw, wd.k16, wd.v16, wd.table16, max_pages, c->num_sms, s,
                                         pdl);
      if (e == cudaSuccess && recon)
        e = rcp::launch_recon<ShapeTiny>(vsrc, c->tmap_wv_mn, p, max_pages, c->num_sms, s, pdl);
      if (e == cudaSuccess)
        e = rcp::launch_prefill<ShapeTiny>(qhi_map, qlo_map, kmap, vals, c->tmap_wv_mn, p,
                                           max_tiles, s, pdl, recon);
    }
    if (e == cudaSuccess && c->prof_stop) e = cudaEventRecord(c->prof_stop, s);
    return e == cudaSuccess ? RCP_OK : RCP_ERR_CUDA;
  }
  p.tile_b = nullptr;   // decode: no prefill tiles, fp32 queries
  p.tile_qt = nullptr;
  p.tcount = nullptr;
  p.qhi = nullptr;
  p.qlo = nullptr;
  // three launches: (A) the step's append with the rank-space queries, (B) the split-K
  // attention, (C) the split-K combine fused with the W_v up-projection (combine.cu)
  CUtensorMap rec_slices, rec_ml;
  if (!(c->shape == kShapeMain ? encode_records<ShapeMain>(&rec_slices, &rec_ml, p.rec, nq)
                               : encode_records<ShapeTiny>(&rec_slices, &rec_ml, p.rec, nq)))
    return RCP_ERR_CUDA;
  rcp_status st2 = launch_front(c, app, q, nq, p.qt, p.qscale, s);
  if (st2 != RCP_OK) return st2;
  rcp::CombineParams cp{};
  cp.cum = p.cum;
  cp.rec = p.rec;
  cp.upart = reinterpret_cast<float*>(
      static_cast<uint8_t*>(ws) +
      (c->shape == kShapeMain ? rcp::ws_layout<ShapeMain>(nq) : rcp::ws_layout<ShapeTiny>(nq)).upart);
  cp.ucnt = p.ucnt;
  cp.out = out;
  cp.dev_err = c->dev_err;
  cp.nq = nq;
  cp.parts = p.parts;
  if (c->shape == kShapeMain) {
    e = rcp::launch_attn<ShapeMain>(c->tmap_v, c->tmap_kpage, p, s, c->prof_start, c->prof_stop);
    if (e == cudaSuccess)
      e = rcp::launch_combine_upproj<ShapeMain>(c->tmap_wv_mn, rec_slices, rec_ml, cp, s, pdl);
  } else {
    e = rcp::launch_attn<ShapeTiny>(c->tmap_v, c->tmap_kpage, p, s, c->prof_start, c->prof_stop);
    if (e == cudaSuccess)
      e = rcp::launch_combine_upproj<ShapeTiny>(c->tmap_wv_mn, rec_slices, rec_ml, cp, s, pdl);
  }
  return e == cudaSuccess ? RCP_OK : RCP_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* rcp_status_string(rcp_status s) {
  switch (s) {
    case RCP_OK: return "ok";
    case RCP_ERR_INVALID_ARG: return "invalid argument";
    case RCP_ERR_UNSUPPORTED: return "unsupported shape";
    case RCP_ERR_CAPACITY: return "block pool capacity / block id error";
    case RCP_ERR_WORKSPACE: return "workspace too small";
    case RCP_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

rcp_status rcp_config_supported(const rcp_cache_config* cfg) {
  if (!cfg) return RCP_ERR_INVALID_ARG;
  if (cfg->page_format != RCP_PAGES_FP16 && cfg->page_format != RCP_PAGES_FP8_E4M3 &&
      cfg->page_format != RCP_PAGES_INT4)
    return RCP_ERR_UNSUPPORTED;
  return shape_of(cfg) == kShapeNone ? RCP_ERR_UNSUPPORTED : RCP_OK;
}

rcp_status rcp_create_cache(const rcp_cache_config* cfg, void* k_pages, void* v_pages,
                            const void* U_k, const void* W_v, uint32_t* dev_error,
                            rcp_cache** out) {
  if (!cfg || !out) return RCP_ERR_INVALID_ARG;
  *out = nullptr;
  if (cfg->num_blocks < 1 || cfg->num_blocks > (int64_t{1} << 26)) return RCP_ERR_INVALID_ARG;
  const int sh = shape_of(cfg);
  if (sh == kShapeNone || rcp_config_supported(cfg) != RCP_OK) return RCP_ERR_UNSUPPORTED;
  if (!k_pages || !v_pages || !U_k || !W_v || !dev_error) return RCP_ERR_INVALID_ARG;
  if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(U_k) || !aligned16(W_v) ||
      (reinterpret_cast<uintptr_t>(dev_error) & 3u))
    return RCP_ERR_INVALID_ARG;
  rcp_cache* c = new (std::nothrow) rcp_cache();
  if (!c) return RCP_ERR_CAPACITY;
  c->cfg = *cfg;
  c->k_pages = k_pages;
  c->v_pages = v_pages;
  c->U_k = U_k;
  c->W_v = W_v;
  c->dev_err = dev_error;
  c->shape = sh;
  c->device = -1;
  c->num_sms = 0;
  c->prof_start = nullptr;
  c->prof_stop = nullptr;
  try {
    c->free_ids.resize(static_cast<size_t>(cfg->num_blocks));
    c->is_free.assign(static_cast<size_t>(cfg->num_blocks), 1);
  } catch (...) {
    delete c;
    return RCP_ERR_CAPACITY;
  }
  // pop order hands out ids 0, 1, 2, ... first
  for (int64_t i = 0; i < cfg->num_blocks; ++i)
    c->free_ids[static_cast<size_t>(i)] = static_cast<int32_t>(cfg->num_blocks - 1 - i);
  *out = c;
  return RCP_OK;
}

rcp_status rcp_destroy_cache(rcp_cache* cache) {
  if (!cache) return RCP_ERR_INVALID_ARG;
  delete cache;
  return RCP_OK;
}

rcp_status rcp_alloc_blocks(rcp_cache* c, int32_t n, int32_t* ids_out) {
  if (!c || n < 0 || (n > 0 && !ids_out)) return RCP_ERR_INVALID_ARG;
  if (static_cast<size_t>(n) > c->free_ids.size()) return RCP_ERR_CAPACITY;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = c->free_ids.back();
    c->free_ids.pop_back();
    c->is_free[static_cast<size_t>(id)] = 0;
    ids_out[i] = id;
  }
  return RCP_OK;
}

rcp_status rcp_free_blocks(rcp_cache* c, int32_t n, const int32_t* ids) {
  if (!c || n < 0 || (n > 0 && !ids)) return RCP_ERR_INVALID_ARG;
  // validate all first so a bad list changes nothing (duplicates inside the list too)
  std::vector<uint8_t> seen;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= c->cfg.num_blocks || c->is_free[static_cast<size_t>(id)])
      return RCP_ERR_CAPACITY;
  }
  if (n > 1) {
    seen.assign(static_cast<size_t>(c->cfg.num_blocks), 0);
    for (int32_t i = 0; i < n; ++i) {
      if (seen[static_cast<size_t>(ids[i])]) return RCP_ERR_CAPACITY;
      seen[static_cast<size_t>(ids[i])] = 1;
    }
  }
  for (int32_t i = 0; i < n; ++i) {
    c->is_free[static_cast<size_t>(ids[i])] = 1;
    c->free_ids.push_back(ids[i]);
  }
  return RCP_OK;
}

rcp_status rcp_num_free_blocks(const rcp_cache* c, int64_t* n_free) {
  if (!c || !n_free) return RCP_ERR_INVALID_ARG;
  *n_free = static_cast<int64_t>(c->free_ids.size());
  return RCP_OK;
}

rcp_status rcp_workspace_size(const rcp_cache* c, int32_t max_query_rows, size_t* bytes) {
  if (!c || !bytes || max_query_rows < 0) return RCP_ERR_INVALID_ARG;
  *bytes = ws_bytes(c, max_query_rows);
  return RCP_OK;
}

rcp_status rcp_append_kv(rcp_cache* c, const void* k, const void* v, const int64_t* slot_mapping,
                         int32_t num_tokens, rcp_stream stream) {
  if (!c || num_tokens < 0) return RCP_ERR_INVALID_ARG;
  if (num_tokens == 0) return RCP_OK;
  const AppendArgs app{k, v, slot_mapping, num_tokens};
  if (check_append(app) != RCP_OK) return RCP_ERR_INVALID_ARG;
  rcp_status st = ensure_device(c);
  if (st != RCP_OK) return st;
  return launch_front(c, &app, nullptr, 0, nullptr, 0.f, static_cast<cudaStream_t>(stream));
}

rcp_status rcp_decode_step(rcp_cache* c, const void* k, const void* v, const int64_t* slot_mapping,
                           int32_t num_tokens, const void* q, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                           void* out, void* workspace, size_t workspace_bytes,
                           rcp_stream stream) {
  if (!c || batch < 0 || num_tokens < 0 || max_blocks_per_seq < 1) return RCP_ERR_INVALID_ARG;
  const AppendArgs app{k, v, slot_mapping, num_tokens};
  return run_attention(c, q, nullptr, batch, block_table, max_blocks_per_seq, seq_lens, batch, out,
                       workspace, workspace_bytes, stream, &app);
}

rcp_status rcp_decode_attn(rcp_cache* c, const void* q, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                           void* out, void* workspace, size_t workspace_bytes,
                           rcp_stream stream) {
  return run_attention(c, q, nullptr, batch, block_table, max_blocks_per_seq, seq_lens, batch, out,
                       workspace, workspace_bytes, stream);
}

rcp_status rcp_decode_attn_sparse(rcp_cache* c, const void* q, const int32_t* block_table,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t batch, float skip_threshold, uint8_t* page_kept,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  rcp_stream stream) {
  if (!(skip_threshold >= 0.f && skip_threshold < 1.f)) return RCP_ERR_INVALID_ARG;   // NaN too
  // weight ratio 2^(s - m) < threshold  <=>  s < m - (-log2 threshold)
  SparseArgs sp{skip_threshold > 0.f ? static_cast<float>(-std::log2(static_cast<double>(skip_threshold)))
                                     : INFINITY,
                page_kept};
  return run_attention(c, q, nullptr, batch, block_table, max_blocks_per_seq, seq_lens, batch, out,
                       workspace, workspace_bytes, stream, nullptr, false, &sp);
}

rcp_status rcp_prefill_attn(rcp_cache* c, const void* q, const int32_t* cu_chunk_lens,
                            int32_t num_query_rows, const int32_t* block_table,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                            void* out, void* workspace, size_t workspace_bytes,
                            rcp_stream stream) {
  if (!cu_chunk_lens) return RCP_ERR_INVALID_ARG;
  return run_attention(c, q, cu_chunk_lens, num_query_rows, block_table, max_blocks_per_seq,
                       seq_lens, batch, out, workspace, workspace_bytes, stream);
}

rcp_status rcp_prefill_attn_reconstruct(rcp_cache* c, const void* q, const int32_t* cu_chunk_lens,
                                        int32_t num_query_rows, const int32_t* block_table,
                                        int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                        int32_t batch, void* out, void* workspace,
                                        size_t workspace_bytes, rcp_stream stream) {
  if (!cu_chunk_lens) return RCP_ERR_INVALID_ARG;
  return run_attention(c, q, cu_chunk_lens, num_query_rows, block_table, max_blocks_per_seq,
                       seq_lens, batch, out, workspace, workspace_bytes, stream, nullptr, true);
}

rcp_status rcp_prefill_step(rcp_cache* c, const void* k, const void* v,
                            const int64_t* slot_mapping, int32_t num_tokens, const void* q,
                            const int32_t* cu_chunk_lens, int32_t num_query_rows,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t batch, int32_t reconstruct,
                            void* out, void* workspace, size_t workspace_bytes,
                            rcp_stream stream) {
  if (!cu_chunk_lens || num_tokens < 0 || (reconstruct != 0 && reconstruct != 1))
    return RCP_ERR_INVALID_ARG;
  const AppendArgs app{k, v, slot_mapping, num_tokens};
  return run_attention(c, q, cu_chunk_lens, num_query_rows, block_table, max_blocks_per_seq,
                       seq_lens, batch, out, workspace, workspace_bytes, stream, &app,
                       reconstruct != 0);
}

rcp_status rcp_prefill_reconstruct_workspace_size(const rcp_cache* c, int32_t max_query_rows,
                                                  int32_t batch, int32_t max_blocks_per_seq,
                                                  size_t* bytes) {
  if (!c || !bytes || max_query_rows < 0 || batch < 0 || max_blocks_per_seq < 0)
    return RCP_ERR_INVALID_ARG;
  *bytes = recon_ws_bytes(c, max_query_rows, batch, max_blocks_per_seq);
  return RCP_OK;
}

rcp_status rcp_prefill_crossover_rows(const rcp_cache* c, int32_t* rows) {
  if (!c || !rows) return RCP_ERR_INVALID_ARG;
  const int64_t R = c->cfg.rank_v, d = c->cfg.head_dim;
  // equal multiply-adds per (key, head): rows * R (rank space) = R * d + rows * d
  *rows = R > d ? static_cast<int32_t>((R * d + (R - d) - 1) / (R - d)) : INT32_MAX;
  return RCP_OK;
}

rcp_status rcp_set_profile_events(rcp_cache* c, void* start_event, void* stop_event) {
  if (!c || ((start_event == nullptr) != (stop_event == nullptr))) return RCP_ERR_INVALID_ARG;
  c->prof_start = static_cast<cudaEvent_t>(start_event);
  c->prof_stop = static_cast<cudaEvent_t>(stop_event);
  return RCP_OK;
}

}  // extern "C"
