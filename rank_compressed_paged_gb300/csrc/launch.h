// Host-side entry points of the kernel translation units (called by the C ABI layer).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "shape.h"

namespace rcp {

template <class S>
cudaError_t prepare_attn(int device);
// The decode's split-K attention kernel (plans its own work from seq_lens; reads the
// rank-space queries the launch before it wrote).
template <class S>
cudaError_t launch_attn(const CUtensorMap& tmap_v, const CUtensorMap& tmap_k, const AttnParams& p,
                        cudaStream_t stream, cudaEvent_t prof_start, cudaEvent_t prof_stop);
// The prefill plan (the prefill path's first kernel).
template <class S>
cudaError_t launch_plan(const AttnParams& p, cudaStream_t stream, bool pdl);
template <class S>
cudaError_t prepare_prefill();
// recon: attend reconstructed values (vp = tensor map of V^, w unused) instead of joint
// coefficients.
template <class S>
cudaError_t launch_prefill(const CUtensorMap& qhi, const CUtensorMap& qlo, const CUtensorMap& kp,
                           const CUtensorMap& vp, const CUtensorMap& w, const AttnParams& p,
                           int max_tiles, cudaStream_t stream, bool pdl, bool recon);
// V^ = C_v W_v for the pages of every request with chunk rows (max_pages bounds them), by
// persistent CTA pairs (at most num_sms / 2).
template <class S>
cudaError_t prepare_recon();
template <class S>
cudaError_t launch_recon(const CUtensorMap& vp, const CUtensorMap& w_v_mn, const AttnParams& p,
                         int64_t max_pages, int num_sms, cudaStream_t stream, bool pdl);
// E4M3 pages: fp16 copies of the batch's pages (plan order) and the re-addressed table.
template <class S>
cudaError_t launch_widen(const AttnParams& p, void* k16, void* v16, int32_t* table16,
                         int64_t max_pages, int num_sms, cudaStream_t stream, bool pdl);
template <class S>
cudaError_t prepare_gemm();
// The append (k_rows / v_rows: tensor maps over the new tokens' k and v, [T][H*d]) and,
// when p.nq > 0, the decode's rank-space queries (q_rows over [nq][H*d]) in one launch;
// boxes 64 x NT with NT = 16 when max(T, nq) <= 16, 64 when it is <= 256, else 256.
template <class S>
cudaError_t launch_append_gemm(const CUtensorMap& w_v, const CUtensorMap& u_k,
                               const CUtensorMap& v_rows, const CUtensorMap& k_rows,
                               const CUtensorMap& q_rows, const AppendParams& p,
                               cudaStream_t stream);
// Prefill rank-space queries on tensor cores (q_rows: [nq][H*d] fp16, boxes 64 x 64 when
// nq <= 256, else 64 x 256).
template <class S>
cudaError_t launch_qproj_gemm(const CUtensorMap& u_k, const CUtensorMap& q_rows, void* qhi,
                              void* qlo, int nq, float qscale, uint32_t* dev_err,
                              cudaStream_t stream, bool pdl);
// Split-K combine fused with the W_v up-projection (combine.cu).  rec_slices / rec_ml: fp32
// tensor maps over the records [(nq + kMaxParts)][REC] with boxes of CombineCfg::CHUNK rows
// by RANKS floats / of REC_ROWS rows by 4 floats.
template <class S>
cudaError_t prepare_combine();
template <class S>
cudaError_t launch_combine_upproj(const CUtensorMap& w_v_mn, const CUtensorMap& rec_slices,
                                  const CUtensorMap& rec_ml, const CombineParams& p,
                                  cudaStream_t stream, bool pdl);

}  // namespace rcp
