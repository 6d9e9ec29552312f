/*
 * rcp.h -- C ABI of the rank-compressed paged attention library (GB300, sm_103a).
 *
 * The method (Proxima page, STAR-KV plugin for vLLM, intro paragraph): keys are kept as
 * per-head low-rank coefficients c_k[t,h] = U_k,h k_{t,h} (r_k numbers per token and
 * head, U_k,h an r_k x d factor with orthonormal rows), values as one joint coefficient
 * vector per token c_v[t] = W_v v_t (R numbers, W_v an R x (H*d) factor), in a paged
 * cache of fixed-size blocks.  Attention runs in rank space:
 *     q~_h = U_k,h q_h,   s_{h,t} = q~_h . c_k[t,h] / sqrt(d),   p_h = softmax(s_h),
 *     z_h = sum_t p_{h,t} c_v[t],   o_h = W_v[:, h*d:(h+1)*d]^T z_h.
 *
 * Memory layout (all device buffers are owned by the caller; the library never
 * allocates device memory; every pointer must be 16-byte aligned):
 *     K pages   [num_blocks][H][block_size][r_k]   fp16 (or E4M3 bytes; 4-bit pages: see
 *                                                  RCP_PAGES_INT4)
 *     V pages   [num_blocks][block_size][R]        fp16 (or E4M3 bytes; 4-bit pages)
 *     U_k       [H][r_k][d]                        fp16
 *     W_v       [R][H*d]   (column h*d + j = head h, element j)   fp16
 *     q, out    [rows][H][d]                       fp16
 *     block_table [rows_of_table][max_blocks_per_seq] int32, physical block ids
 *     seq_lens  [batch] int32 (tokens in the cache, including any just appended)
 * Token t of a request lives in block block_table[b][t / block_size] at offset
 * t % block_size; a slot id is block * block_size + offset (vLLM convention).
 *
 * Errors: host-checkable problems (null or misaligned pointers, bad sizes, unsupported
 * shapes, a workspace that is too small) return a status synchronously and launch
 * nothing.  Values that live on the device (slots, block ids, lengths) are checked by the
 * kernels: a bad value sets a bit in the caller-provided device error word
 * (RCP_DEVERR_*) and the offending slot / block contributes nothing.  Launch failures
 * return RCP_ERR_CUDA.  No call synchronises the host; all work is queued on the given
 * stream.  No C++ exception crosses this interface.
 */
#ifndef RCP_H_
#define RCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rcp_status {
  RCP_OK = 0,
  RCP_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, negative or inconsistent size */
  RCP_ERR_UNSUPPORTED = 2,   /* shape this build has no kernel for */
  RCP_ERR_CAPACITY = 3,      /* block pool exhausted / id out of range / double free */
  RCP_ERR_WORKSPACE = 4,     /* workspace smaller than rcp_workspace_size() */
  RCP_ERR_CUDA = 5           /* a CUDA runtime / driver call failed */
} rcp_status;

/* Bits a kernel ORs into the device error word. */
#define RCP_DEVERR_BAD_SLOT 1u    /* append: slot >= num_blocks * block_size */
#define RCP_DEVERR_BAD_BLOCK 2u   /* attention: block id outside [0, num_blocks) */
#define RCP_DEVERR_BAD_LEN 4u     /* attention: seq_len < 0, > table capacity, or chunk > seq_len */
#define RCP_DEVERR_TIMEOUT 8u     /* a pipeline wait exceeded its bound; results invalid */

/* Element type of the K and V pages. */
#define RCP_PAGES_FP16 0      /* IEEE fp16 coefficients */
#define RCP_PAGES_FP8_E4M3 1  /* E4M3 codes (OCP 8-bit float: bias 7, 3 mantissa bits, max
                                 448): the append rounds to nearest even and saturates to
                                 +-448; half the bytes per token.  Append, decode (dense
                                 and block-sparse) and both prefill variants (pages
                                 widened to fp16 first). */
#define RCP_PAGES_INT4 2      /* 4-bit codes with fp16 scales ("KV-cache LLM serving" page,
                                 "What it measured", item 1: 4-bit KV pages for capacity;
                                 a rotation before quantizing folds into U_k and W_v, so it
                                 needs no call of its own).  One K page is
                                 H*16*r_k/2 bytes of codes (key row (h, t) at byte
                                 (h*16 + t)*r_k/2, two per byte, even index in the low
                                 nibble, two's complement in [-7, 7]) then H*16 fp16 scales
                                 (row (h, t) at index h*16 + t); one V page is 16*R/2 bytes
                                 of codes (token t at byte t*R/2) then 16*(R/64) fp16 scales
                                 (token t, group g of 64 coefficients at index t*(R/64)+g).
                                 A coefficient is code * scale.  The append accumulates in
                                 fp32 and per group (a key row; 64 value coefficients) takes
                                 the smallest fp16 scale with 7*scale >= max|x| and
                                 code = x/scale rounded to nearest, ties to even.  The
                                 decode widens value coefficients to fp16(code * scale)
                                 (one rounding) and scores keys as scale * (codes . q~) in
                                 fp32.  1,632 bytes per token at (32, 128, 64, 1024).
                                 Append, decode (dense and block-sparse) and both prefill
                                 variants (which widen K and V to fp16(code * scale)
                                 first). */

typedef struct rcp_cache_config {
  int32_t num_heads;   /* H */
  int32_t head_dim;    /* d */
  int32_t rank_k;      /* r_k, key coefficients per token and head */
  int32_t rank_v;      /* R, joint value coefficients per token */
  int32_t block_size;  /* tokens per page; this build supports 16 */
  int64_t num_blocks;  /* physical blocks in the K and V page buffers */
  int32_t page_format; /* RCP_PAGES_FP16, RCP_PAGES_FP8_E4M3 or RCP_PAGES_INT4 */
} rcp_cache_config;

typedef struct rcp_cache rcp_cache;   /* opaque handle: borrowed pointers + host free list */
typedef void* rcp_stream;             /* a cudaStream_t; NULL means the legacy stream */

/* Human-readable name of a status code (static string). */
const char* rcp_status_string(rcp_status s);

/* RCP_OK if this build has kernels for the shape.  Supported: block_size 16 and
 * (H, d, r_k, R) = (32, 128, 64, 1024) or (4, 64, 16, 64). */
rcp_status rcp_config_supported(const rcp_cache_config* cfg);

/* Create a handle over caller-owned device buffers (layout above): the compressed paged
 * cache of the Proxima page (STAR-KV plugin for vLLM), intro paragraph, which keeps the
 * per-head key coefficients and the joint value coefficients in fixed-size pages and
 * holds the factors U_k and W_v beside them.  dev_error points to one device uint32 the
 * kernels OR error bits into (the caller zeroes and reads it).  Makes no CUDA call; the
 * handle's host free list starts with all blocks free.
 * Errors: RCP_ERR_UNSUPPORTED for a shape or page format without kernels;
 * RCP_ERR_INVALID_ARG for a null or misaligned pointer or num_blocks outside [1, 2^26].
 * Ownership: the caller keeps every buffer alive until rcp_destroy_cache, which frees only
 * the handle's host memory (never the caller's buffers). */
rcp_status rcp_create_cache(const rcp_cache_config* cfg, void* k_pages, void* v_pages,
                            const void* U_k, const void* W_v, uint32_t* dev_error,
                            rcp_cache** out);
rcp_status rcp_destroy_cache(rcp_cache* cache);

/* Host-side block pool: capacity accounting for the paged cache, in the unit the Proxima
 * page counts capacity in ("KV-cache capacity": GPU KV blocks that fit the same memory
 * budget).  alloc hands out n free physical ids into ids_out[0..n) (host array, caller
 * owned; RCP_ERR_CAPACITY and no change if fewer are free); free returns n ids from a
 * host array (RCP_ERR_CAPACITY and no change on an out-of-range, already-free or repeated
 * id); num_free reports the free count.  Pure host bookkeeping, no CUDA call; a handle is
 * not thread-safe. */
rcp_status rcp_alloc_blocks(rcp_cache* cache, int32_t n, int32_t* ids_out);
rcp_status rcp_free_blocks(rcp_cache* cache, int32_t n, const int32_t* ids);
rcp_status rcp_num_free_blocks(const rcp_cache* cache, int64_t* n_free);

/* Bytes of device workspace decode / prefill need for up to max_query_rows query rows
 * (decode: batch; prefill: total chunk rows): the split-K partial records of the
 * "Per-decode-step attention" section's split attention and its combine step (Proxima
 * page, "Kernel profiling breakdown", the combine-splits kernel), the plan and the
 * rank-space queries.  The caller allocates it (256-byte aligned) and may reuse it for
 * every call on one stream.  Pure host arithmetic; RCP_ERR_INVALID_ARG for a null
 * handle or output, or a negative row count. */
rcp_status rcp_workspace_size(const rcp_cache* cache, int32_t max_query_rows, size_t* bytes);

/* Append (Proxima page, "Kernel profiling breakdown": the cache-write kernel does the
 * low-rank projection): for each of num_tokens new tokens i with slot s =
 * slot_mapping[i] >= 0, write fp16(U_k,h k[i][h]) to K page [s/bs][h][s%bs] for every
 * head and fp16(W_v v[i]) (v[i] flattened head-major) to V page [s/bs][s%bs].  slot -1
 * is skipped.  Each coefficient is accumulated in fp32 and rounded once to the page format,
 * to nearest with ties to even (fp16 pages; E4M3 pages also saturate at +-448).
 * k, v: [num_tokens][H][d] fp16 device; slot_mapping: [num_tokens] int64 device.
 * Duplicate slots within one call are undefined. */
rcp_status rcp_append_kv(rcp_cache* cache, const void* k, const void* v,
                         const int64_t* slot_mapping, int32_t num_tokens, rcp_stream stream);

/* Decode attention (Proxima page, "Per-decode-step attention"): one query per request,
 * q [batch][H][d] fp16, attends the first seq_lens[b] tokens of request b through
 * block_table row b.  out [batch][H][d] fp16; seq_len 0 gives zeros.  workspace must hold
 * rcp_workspace_size(cache, batch) bytes (256-byte aligned); its contents are scratch. */
rcp_status rcp_decode_attn(rcp_cache* cache, const void* q, const int32_t* block_table,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                           void* out, void* workspace, size_t workspace_bytes,
                           rcp_stream stream);

/* Block-sparse decode ("KV-cache LLM serving" page, "What it measured", item 3: decode
 * kernels that skip low-weight blocks using the online softmax).  Same arguments and
 * result as rcp_decode_attn, except that a page is left out when, for every head, its
 * largest softmax weight is below skip_threshold times the largest weight that head has
 * met so far in the pass: its value coefficients are not read and its tokens take part
 * in neither the softmax numerator nor its denominator.  Keys are always read (scores
 * decide).  Value coefficients are shared by all heads, so a page is read when any head
 * needs it.  The pass keeps one running maximum per work partition (a partition starts
 * with its first page kept), so which pages are left out depends on how the batch is
 * partitioned; every page left out satisfies the rule against the running maximum, which
 * never exceeds the maximum over the whole sequence.
 *   skip_threshold: in [0, 1); 0 leaves no page out; otherwise RCP_ERR_INVALID_ARG.
 *     With 0 the result is that of rcp_decode_attn bit for bit on fp16 pages, and on
 *     quantized pages where the dense decode also scores keys on the CUDA cores (r_k != 64
 *     or H % 16 != 0); elsewhere the dense decode scores E4M3 and 4-bit keys on the tensor
 *     cores and the two agree to rounding.
 *   page_kept: NULL, or device uint8 [batch][max_blocks_per_seq]: entry (b, j) is set to 1
 *     if page j of request b was read and 0 if it was left out; entries at or past
 *     ceil(seq_lens[b] / 16) are not written.
 * Every page format: E4M3 and 4-bit keys are scored on the CUDA cores here (a page's
 * value codes are widened only once the page is kept).  Workspace as rcp_decode_attn. */
rcp_status rcp_decode_attn_sparse(rcp_cache* cache, const void* q, const int32_t* block_table,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t batch, float skip_threshold, uint8_t* page_kept,
                                  void* out, void* workspace, size_t workspace_bytes,
                                  rcp_stream stream);

/* One decode step: rcp_append_kv(k, v, slot_mapping, num_tokens) followed by
 * rcp_decode_attn(q, ...), with the same arguments and results (the pages' "per-decode-step"
 * unit: the cache write and the attention of a step).  Queued together, the query
 * projection of the attention runs alongside the append (it reads nothing the append
 * writes), which shortens the step.  All checks of both calls apply before anything is
 * launched except the append's own. */
rcp_status rcp_decode_step(rcp_cache* cache, const void* k, const void* v,
                           const int64_t* slot_mapping, int32_t num_tokens, const void* q,
                           const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t batch, void* out, void* workspace,
                           size_t workspace_bytes, rcp_stream stream);

/* Chunked-prefill attention (Proxima page, "Per-prefill-chunk attention").  The chunk's
 * K/V must already be appended.  Request b owns query rows cu_chunk_lens[b] ..
 * cu_chunk_lens[b+1]-1 of q [num_query_rows][H][d]; seq_lens[b] counts prior + chunk
 * tokens; chunk row i sits at position seq_lens[b] - chunk_b + i and attends keys
 * 0 .. that position (causal).  cu_chunk_lens must not decrease: if any entry is below
 * the one before it, RCP_DEVERR_BAD_LEN is set and no row of out is written (so that no
 * two requests can claim the same rows).  out [num_query_rows][H][d] fp16.  workspace must hold
 * rcp_workspace_size(cache, num_query_rows) bytes; on E4M3 and 4-bit pages, which are first
 * widened to fp16 in the workspace as for rcp_prefill_attn_reconstruct, it must hold
 * rcp_prefill_reconstruct_workspace_size(cache, num_query_rows, batch,
 * max_blocks_per_seq) bytes. */
rcp_status rcp_prefill_attn(rcp_cache* cache, const void* q, const int32_t* cu_chunk_lens,
                            int32_t num_query_rows, const int32_t* block_table,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch,
                            void* out, void* workspace, size_t workspace_bytes,
                            rcp_stream stream);

/* Chunked prefill, reconstructing variant (Proxima page, "Per-prefill-chunk attention",
 * whose prefill kernel expands compressed keys per query tile; here the joint value
 * coefficients are the ones expanded, once per key).  Same arguments, layout and
 * results as rcp_prefill_attn, up to rounding: the values of every cached key of the
 * requests with chunk rows are first reconstructed as V^ = C_v W_v (fp32 accumulation,
 * stored fp16) and the attention then runs on V^ with O = P V^ per head.  Cheaper than
 * the rank-space variant once a request's chunk has more than rcp_prefill_crossover_rows
 * rows.  workspace must hold rcp_prefill_reconstruct_workspace_size(cache, num_query_rows,
 * batch, max_blocks_per_seq) bytes (256-byte aligned; it grows with the pages the batch
 * can reach, 2 * H * d * 16 bytes per page).  E4M3 and 4-bit pages: every page the batch
 * reads is first widened to fp16 in the workspace (E4M3 exactly, 4-bit as fp16(code *
 * scale)), which then also holds 2 * 16 * (H * r_k + R) + 4 bytes per page the batch can
 * reach; the result is that of the same call on fp16 pages holding the widened values. */
rcp_status rcp_prefill_attn_reconstruct(rcp_cache* cache, const void* q,
                                        const int32_t* cu_chunk_lens, int32_t num_query_rows,
                                        const int32_t* block_table, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, int32_t batch, void* out,
                                        void* workspace, size_t workspace_bytes,
                                        rcp_stream stream);

/* A chunked prefill step: rcp_append_kv(k, v, slot_mapping, num_tokens) (the chunk's own
 * keys and values) followed by rcp_prefill_attn (reconstruct = 0) or
 * rcp_prefill_attn_reconstruct (reconstruct = 1) with the remaining arguments, on one
 * stream, with the same results.  Proxima page, "Per-prefill-chunk attention": each chunk
 * row attends its causal prefix, which includes the chunk's own tokens, so a serving step
 * appends them first.  Queued as one step: the chunk's query projection runs in the
 * append's launch, and the plan beside it.  Arguments, layouts, workspace size and errors
 * as the two calls; reconstruct other than 0 or 1 is RCP_ERR_INVALID_ARG; with
 * num_query_rows = 0 only the append runs. */
rcp_status rcp_prefill_step(rcp_cache* cache, const void* k, const void* v,
                            const int64_t* slot_mapping, int32_t num_tokens, const void* q,
                            const int32_t* cu_chunk_lens, int32_t num_query_rows,
                            const int32_t* block_table, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t batch, int32_t reconstruct,
                            void* out, void* workspace, size_t workspace_bytes,
                            rcp_stream stream);

/* Workspace bytes of rcp_prefill_attn_reconstruct. */
rcp_status rcp_prefill_reconstruct_workspace_size(const rcp_cache* cache, int32_t max_query_rows,
                                                  int32_t batch, int32_t max_blocks_per_seq,
                                                  size_t* bytes);

/* Chunk rows per request above which the reconstructing prefill does fewer multiply-adds:
 * ceil(R d / (R - d)) (147 for R = 1024, d = 128); INT32_MAX when R <= d. */
rcp_status rcp_prefill_crossover_rows(const rcp_cache* cache, int32_t* rows);

/* Measurement hook (the pages have no counterpart; it exists for roofline timing).  When
 * both events are non-NULL, every later decode / prefill call records start_event on its
 * stream just before the split-K attention kernel and stop_event just after it, so the
 * caller can read that kernel's duration with cudaEventElapsedTime.  The events are
 * cudaEvent_t handles owned by the caller; NULL, NULL turns the hook off. */
rcp_status rcp_set_profile_events(rcp_cache* cache, void* start_event, void* stop_event);

/* Decode without any caller-provided or allocated device memory.  The paper has no
 * counterpart; this entry point exists for callers that cannot allocate: a host runtime
 * that owns all device memory and gives plugins no workspace, or a serving loop that must
 * not call cudaMalloc after start-up (an allocation can wait on device-wide
 * synchronisation).  Same arguments and result as rcp_decode_attn minus the workspace:
 * the scratch is a fixed array of RCP_NOALLOC_SCRATCH_BYTES inside this library, which
 * every GPU that loads the library holds until the process exits.
 *   - Limit: batch must satisfy rcp_workspace_size(cache, batch) <=
 *     RCP_NOALLOC_SCRATCH_BYTES (for H=32, d=128, r_k=64, R=1024 that is batch <= 157);
 *     a larger batch returns RCP_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address (once per device,
 *     with that device current) and keeps it for the life of the process; make that
 *     first call before any stream capture.  A cudaDeviceReset between calls is not
 *     supported: it unloads the module, and the kept address goes stale.
 *   - Allocates nothing: no cudaMalloc / cudaFree and no allocating library routine.
 *   - Every call shares the one array: calls that overlap on the GPU (other streams,
 *     other threads, no ordering between them) race and give wrong results.  Each call
 *     rewrites all the scratch it reads, so earlier contents never leak into a result. */
#define RCP_NOALLOC_SCRATCH_BYTES (64ull << 20)
rcp_status rcp_decode_attn_noalloc(rcp_cache* cache, const void* q, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                   int32_t batch, void* out, rcp_stream stream);

#ifdef __cplusplus
}
#endif
#endif  /* RCP_H_ */
