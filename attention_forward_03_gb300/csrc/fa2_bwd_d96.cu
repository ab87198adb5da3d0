// Instantiations of the backward kernel at head dimension 96 (in the tiles of 128).
#include "fa2_bwd_kernel.cuh"

namespace fa2 {
template cudaError_t launch_bwd<96, false, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                 const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
template cudaError_t launch_bwd<96, false, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
template cudaError_t launch_bwd<96, true, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
template cudaError_t launch_bwd<96, true, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
}  // namespace fa2
