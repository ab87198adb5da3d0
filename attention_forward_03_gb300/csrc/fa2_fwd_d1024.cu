// Instantiations of the d-tiled sm_103a forward kernel for head dimension 1024.
#include "fa2_kernel_dtile.cuh"

namespace fa2 {
template cudaError_t launch_fwd_dtile<1024, false, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                      const CUtensorMap&, const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_dtile<1024, false, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     const CUtensorMap&, const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_dtile<1024, true, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                     const CUtensorMap&, const Params&, int, cudaStream_t);
template cudaError_t launch_fwd_dtile<1024, true, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                    const CUtensorMap&, const Params&, int, cudaStream_t);
}  // namespace fa2
