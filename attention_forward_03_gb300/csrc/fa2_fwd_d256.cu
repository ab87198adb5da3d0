// Instantiations of the sm_103a forward kernel for head dimension 256.
#include "fa2_kernel_wide.cuh"

namespace fa2 {
template cudaError_t launch_fwd_wide<256, false, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                        const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_wide<256, false, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                       const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_wide<256, true, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                       const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_wide<256, true, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const Params&, int, cudaStream_t);
}  // namespace fa2
