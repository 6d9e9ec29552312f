// Decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: a host runtime that owns
// every byte of device memory and gives its plugins none (an inference engine's custom
// operator hook, for instance), or a latency-critical serving loop that must not call
// cudaMalloc once it is running, because an allocation can stall on device-wide
// synchronisation.  rcp_decode_attn_noalloc serves them: it runs the same kernels as
// rcp_decode_attn, with the scratch taken from a fixed device array that lives in this
// library's module instead of a caller buffer.  It allocates nothing itself.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "rcp.h"

namespace {

// The scratch array.  Every GPU that loads the library holds these bytes until the
// process exits.  In host code this name is only a host-side stand-in for the device
// symbol; kernels receive the device address obtained from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RCP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once per device
// (with that device current) and remembered.
rcp_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RCP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return RCP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return RCP_OK;
}

}  // namespace

extern "C" rcp_status rcp_decode_attn_noalloc(rcp_cache* cache, const void* q,
                                              const int32_t* block_table,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* seq_lens, int32_t batch, void* out,
                                              rcp_stream stream) {
  if (!cache || batch < 0) return RCP_ERR_INVALID_ARG;
  size_t need = 0;
  rcp_status st = rcp_workspace_size(cache, batch, &need);
  if (st != RCP_OK) return st;
  if (need > RCP_NOALLOC_SCRATCH_BYTES) return RCP_ERR_WORKSPACE;   // batch beyond the limit
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != RCP_OK) return st;
  // The kernels write every scratch byte they later read (plan, queries, partials,
  // merged sums), so the previous call's contents need no clearing.
  return rcp_decode_attn(cache, q, block_table, max_blocks_per_seq, seq_lens, batch, out, scratch,
                         RCP_NOALLOC_SCRATCH_BYTES, stream);
}
