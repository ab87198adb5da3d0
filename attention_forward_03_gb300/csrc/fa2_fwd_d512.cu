// Instantiations of the d-tiled sm_103a forward kernel for head dimension 512.
#include "fa2_kernel_dtile.cuh"

namespace fa2 {
template cudaError_t launch_fwd_dtile<512, false, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_dtile<512, false, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     const CUtensorMap&, const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_dtile<512, true, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     const CUtensorMap&, const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_dtile<512, true, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                    const CUtensorMap&, const Params&, int, cudaStream_t);
}  // namespace fa2
