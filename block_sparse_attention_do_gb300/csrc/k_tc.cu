// k_tc.cu -- placeholder until the tensor-core kernels land.
#include "launch.h"

namespace nsa {

bool tc_supported(const Geo &, int) { return false; }

cudaError_t launch_fwd_tc(const Geo &, const void *, const void *, const void *, const int *, void *,
                          float *, int *, cudaStream_t)
{
    return cudaErrorNotSupported;
}
cudaError_t launch_dq_tc(const Geo &, const void *, const void *, const void *, const void *,
                         const float *, const float *, const int *, void *, int *, cudaStream_t)
{
    return cudaErrorNotSupported;
}
cudaError_t launch_dkdv_tc(const Geo &, const void *, const void *, const void *, const void *,
                           const float *, const float *, const int *, const int *, const Unit *,
                           const WsHeader *, int, float *, void *, void *, int *, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace nsa
