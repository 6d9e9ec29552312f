// Append: project new tokens to low-rank coefficients and scatter them into pages.
//
// The cache-write step of the Proxima page ("Kernel profiling breakdown": the write
// kernel does the low-rank projection).  For token i with slot s >= 0:
//   K page [s/16][h][s%16][:] = fp16(U_k,h k_{i,h})   for every head h
//   V page [s/16][s%16][:]    = fp16(W_v v_i)         (v_i flattened head-major)
// fp32 accumulation, round to nearest even.  One launch holds two kinds of CTAs: key
// projection tiles (token tile x head) and value projection tiles (token tile x 64
// joint-rank rows, reduction over H*d staged through shared memory).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "rcp.h"
#include "shape.h"

namespace rcp {

constexpr int kAppThreads = 256;
constexpr int kKTile = 16;    // tokens per key-projection CTA
constexpr int kVTile = 8;     // tokens per value-projection CTA
constexpr int kVRows = 64;    // joint-rank rows per value-projection CTA
constexpr int kVChunk = 64;   // reduction chunk (elements of H*d)

__device__ __forceinline__ bool slot_target(const AppendParams& p, int64_t s, int64_t* blk,
                                            int* off) {
  if (s < 0) return false;
  if (s >= p.num_blocks * kBlockSize) {
    atomicOr(p.dev_err, RCP_DEVERR_BAD_SLOT);
    return false;
  }
  *blk = s / kBlockSize;
  *off = static_cast<int>(s % kBlockSize);
  return true;
}

template <class S>
__global__ void __launch_bounds__(kAppThreads) append_kernel(const AppendParams p, int n_kcta) {
  constexpr int H = S::H, D = S::D, RK = S::RK, R = S::R, HD = S::H * S::D;
  __shared__ float sa[kKTile * (D + 1) > kVTile * kVChunk ? kKTile * (D + 1) : kVTile * kVChunk];
  __shared__ float sb[D * RK > kVChunk * (kVRows + 1) ? D * RK : kVChunk * (kVRows + 1)];
  const int tid = threadIdx.x;
  if (static_cast<int>(blockIdx.x) < n_kcta) {
    // ---------------------------------------------------------------- key projection
    const int h = blockIdx.x % H;
    const int t0 = (blockIdx.x / H) * kKTile;
    float* ks = sa;                      // [kKTile][D + 1]
    float* ut = sb;                      // [D][RK]: ut[j][k] = U[h][k][j]
    const __half* U = static_cast<const __half*>(p.U_k) + static_cast<size_t>(h) * RK * D;
    const __half* K = static_cast<const __half*>(p.k);
    for (int i = tid; i < RK * D; i += kAppThreads) ut[(i % D) * RK + i / D] = __half2float(U[i]);
    for (int i = tid; i < kKTile * D; i += kAppThreads) {
      const int tt = i / D, j = i % D;
      const int tok = t0 + tt;
      ks[tt * (D + 1) + j] =
          tok < p.T ? __half2float(K[(static_cast<size_t>(tok) * H + h) * D + j]) : 0.f;
    }
    __syncthreads();
    constexpr int NG = kAppThreads / RK;
    constexpr int PER = (kKTile + NG - 1) / NG;
    const int k = tid % RK, grp = tid / RK;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int j = 0; j < D; ++j) {
      const float u = ut[j * RK + k];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int tt = grp + i * NG;
        if (tt < kKTile) acc[i] = fmaf(u, ks[tt * (D + 1) + j], acc[i]);
      }
    }
    __half* kp = static_cast<__half*>(p.k_pages);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int tt = grp + i * NG;
      const int tok = t0 + tt;
      if (tt >= kKTile || tok >= p.T) continue;
      int64_t blk;
      int off;
      if (!slot_target(p, p.slots[tok], &blk, &off)) continue;
      kp[((blk * H + h) * kBlockSize + off) * RK + k] = __float2half_rn(acc[i]);
    }
    return;
  }
  // ------------------------------------------------------------------ value projection
  const int vb = blockIdx.x - n_kcta;
  constexpr int NRT = (R + kVRows - 1) / kVRows;
  const int r0 = (vb % NRT) * kVRows;
  const int t0 = (vb / NRT) * kVTile;
  float* vs = sa;                        // [kVTile][kVChunk]
  float* wt = sb;                        // [kVChunk][kVRows + 1]: wt[j][r] = W[r0 + r][j0 + j]
  const __half* V = static_cast<const __half*>(p.v);
  const __half* W = static_cast<const __half*>(p.W_v);
  constexpr int NG = kAppThreads / kVRows;
  constexpr int PER = kVTile / NG;
  const int r = tid % kVRows, grp = tid / kVRows;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int j0 = 0; j0 < HD; j0 += kVChunk) {
    __syncthreads();
    for (int i = tid; i < kVTile * kVChunk; i += kAppThreads) {
      const int tt = i / kVChunk, j = i % kVChunk;
      const int tok = t0 + tt;
      vs[i] = tok < p.T ? __half2float(V[static_cast<size_t>(tok) * HD + j0 + j]) : 0.f;
    }
    for (int i = tid; i < kVRows * kVChunk; i += kAppThreads) {
      const int rr = i / kVChunk, j = i % kVChunk;
      wt[j * (kVRows + 1) + rr] =
          (r0 + rr < R) ? __half2float(W[static_cast<size_t>(r0 + rr) * HD + j0 + j]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int j = 0; j < kVChunk; ++j) {
      const float w = wt[j * (kVRows + 1) + r];
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, vs[(grp + i * NG) * kVChunk + j], acc[i]);
    }
  }
  __half* vp = static_cast<__half*>(p.v_pages);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int tok = t0 + grp + i * NG;
    if (tok >= p.T || r0 + r >= R) continue;
    int64_t blk;
    int off;
    if (!slot_target(p, p.slots[tok], &blk, &off)) continue;
    vp[(blk * kBlockSize + off) * R + r0 + r] = __float2half_rn(acc[i]);
  }
}

template <class S>
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  const int n_kcta = ((p.T + kKTile - 1) / kKTile) * S::H;
  const int n_vcta = ((p.T + kVTile - 1) / kVTile) * ((S::R + kVRows - 1) / kVRows);
  append_kernel<S><<<n_kcta + n_vcta, kAppThreads, 0, stream>>>(p, n_kcta);
  return cudaGetLastError();
}

template cudaError_t launch_append<ShapeMain>(const AppendParams&, cudaStream_t);
template cudaError_t launch_append<ShapeTiny>(const AppendParams&, cudaStream_t);

}  // namespace rcp
