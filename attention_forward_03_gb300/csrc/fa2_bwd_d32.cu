// Instantiations of the backward kernel at head dimension 32 (in the tiles of 64).
#include "fa2_bwd_kernel.cuh"

namespace fa2 {
template cudaError_t launch_bwd<32, false, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                 const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
template cudaError_t launch_bwd<32, false, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
template cudaError_t launch_bwd<32, true, false>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
template cudaError_t launch_bwd<32, true, true>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                               const CUtensorMap&, const CUtensorMap&, const BwdParams&, int,
                                                 cudaStream_t);
}  // namespace fa2
