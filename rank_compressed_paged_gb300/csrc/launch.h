// Host-side entry points of the kernel translation units (called by the C ABI layer).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "shape.h"

namespace rcp {

template <class S>
cudaError_t prepare_attn(int device);
template <class S>
cudaError_t launch_attn(const CUtensorMap& tmap_v, const AttnParams& p, cudaStream_t stream,
                        cudaEvent_t prof_start, cudaEvent_t prof_stop);
template <class S>
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

}  // namespace rcp
