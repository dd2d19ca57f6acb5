// Host entry points of the bulk-copy convert_combine_input (ep_convert.cu).
#pragma once

#include "ep_kernels.cuh"

namespace ep {

// convert_combine_input through the bulk-copy ring: top-k <= 8.
bool convert_combine_bulk_supported(const ConvertParams& p);
cudaError_t launch_convert_combine_bulk(const ConvertParams& p, int dtype, const LaunchCfg& lc,
                                        cudaStream_t st);

}  // namespace ep
